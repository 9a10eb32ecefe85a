"""Host memory at the edges of a step: sfa_copy_cache_rows places rows from page-locked host
memory (or the device) into strided cache slots, and the attention entry points write O and
lse straight into page-locked host memory -- bit for bit what they write on the device."""
import pytest
import torch

from test_gpu_pipeline import _check_queries, _run, _step_for

pytestmark = pytest.mark.gpu

sfa = pytest.importorskip("indexer_selected_sparse_block_gb300")


@pytest.fixture(scope="module")
def dev():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()
    return torch.device("cuda:0")


@pytest.mark.parametrize("src_on", ["host", "device"])
@pytest.mark.parametrize("n_new", [1, 3])
def test_copy_cache_rows_into_strided_slots(dev, src_on, n_new):
    g = torch.Generator().manual_seed(11)
    cache = torch.randn((5, 40, 2, 72), generator=g).to(torch.bfloat16).to(dev)
    before = cache.clone()
    rows = torch.randn((5, n_new, 2, 72), generator=g).to(torch.bfloat16)
    src = rows.pin_memory() if src_on == "host" else rows.to(dev)
    sfa.sfa_copy_cache_rows(cache[:, 17:17 + n_new], src)
    torch.cuda.synchronize()
    assert torch.equal(cache[:, 17:17 + n_new].cpu(), rows)
    assert torch.equal(cache[:, :17], before[:, :17])            # nothing else moved
    assert torch.equal(cache[:, 17 + n_new:], before[:, 17 + n_new:])


@pytest.mark.parametrize("src_on", ["host", "device"])
def test_copy_cache_rows_odd_sizes(dev, src_on):
    """Rows whose size and pitches are not multiples of 16 bytes (the byte-wise path), and one
    long row (a step's query inputs as one copy)."""
    g = torch.Generator().manual_seed(12)
    cache = torch.randint(-100, 100, (4, 10, 15), generator=g, dtype=torch.int8).to(dev)
    before = cache.clone()
    rows = torch.randint(-100, 100, (4, 1, 15), generator=g, dtype=torch.int8)
    src = rows.pin_memory() if src_on == "host" else rows.to(dev)
    sfa.sfa_copy_cache_rows(cache[:, 7:8], src)
    torch.cuda.synchronize()
    assert torch.equal(cache[:, 7:8].cpu(), rows)
    assert torch.equal(cache[:, :7], before[:, :7]) and torch.equal(cache[:, 8:], before[:, 8:])
    big = torch.randint(0, 255, (1, 700000), generator=g, dtype=torch.uint8)
    big_src = big.pin_memory() if src_on == "host" else big.to(dev)
    dst = torch.zeros((1, 700000), dtype=torch.uint8, device=dev)
    sfa.sfa_copy_cache_rows(dst, big_src)
    torch.cuda.synchronize()
    assert torch.equal(dst.cpu(), big)


def test_copy_cache_rows_multi(dev):
    """Three copies in one launch -- one long row, strided bf16 rows, odd-sized int8 rows --
    each lands where the single copy puts it."""
    g = torch.Generator().manual_seed(13)
    arena_h = torch.randint(0, 255, (1, 123456), generator=g, dtype=torch.uint8).pin_memory()
    arena_d = torch.zeros((1, 123456), dtype=torch.uint8, device=dev)
    K = torch.zeros((6, 30, 1, 576), dtype=torch.bfloat16, device=dev)
    krows = torch.randn((6, 1, 1, 576), generator=g).to(torch.bfloat16).pin_memory()
    X = torch.zeros((6, 30, 15), dtype=torch.int8, device=dev)
    xrows = torch.randint(-9, 9, (6, 1, 15), generator=g, dtype=torch.int8).pin_memory()
    sfa.sfa_copy_cache_rows_multi([(arena_d, arena_h), (K[:, 29:30], krows), (X[:, 4:5], xrows)])
    torch.cuda.synchronize()
    assert torch.equal(arena_d.cpu(), arena_h)
    assert torch.equal(K[:, 29:30].cpu(), krows) and torch.count_nonzero(K[:, :29]) == 0
    assert torch.equal(X[:, 4:5].cpu(), xrows) and torch.count_nonzero(X[:, 5:]) == 0


def test_copy_cache_rows_rejects_unpinned_and_mismatched(dev):
    cache = torch.zeros((4, 8, 16), dtype=torch.bfloat16, device=dev)
    with pytest.raises(ValueError):
        sfa.sfa_copy_cache_rows(cache[:, 2], torch.zeros((4, 16), dtype=torch.bfloat16))
    with pytest.raises(ValueError):
        sfa.sfa_copy_cache_rows(cache[:, 2], torch.zeros((4, 15), dtype=torch.bfloat16,
                                                           device=dev))


@pytest.mark.parametrize("name", ["decode_1x4096", "decode_32x131072"])
def test_attention_writes_host_output(dev, name):
    """sfa_gather_attend with O and lse in page-locked host memory gives the device call's
    bits."""
    w = sfa.WORKLOADS[name]
    w = w.with_(n_seq=3) if name == "decode_1x4096" else w
    case, step = _run(w, dev)
    O_host = torch.empty(step.O.shape, dtype=torch.float32).pin_memory()
    lse_host = torch.empty(step.lse.shape, dtype=torch.float32).pin_memory()
    sfa.sfa_gather_attend(case["Q"], case["K"], case["V"], case["q_seq"], case["q_pos"],
                          step.blk_idx, step.n_sel, step.top_k, w.compress_ratio, w.scale,
                          O_host, lse=lse_host, workspace=step.attn_ws, dev_status=step.status)
    torch.cuda.synchronize()
    assert sfa.sfa_read_device_status(step.status) == 0
    assert torch.equal(O_host, step.O.cpu())
    assert torch.equal(lse_host, step.lse.cpu())
    with pytest.raises(ValueError):   # pageable host memory is refused
        sfa.sfa_gather_attend(case["Q"], case["K"], case["V"], case["q_seq"], case["q_pos"],
                              step.blk_idx, step.n_sel, step.top_k, w.compress_ratio, w.scale,
                              torch.empty(step.O.shape, dtype=torch.float32))


@pytest.mark.parametrize("window_mode", ["single", "split"])
def test_step_output_in_host_memory(dev, window_mode):
    """SfaStep.set_output routes O to page-locked host memory; with a dense window in either
    mode the host result is the device result and matches the oracle."""
    w = sfa.WORKLOADS["decode_1x4096"].with_(n_seq=4)
    case = sfa.make_case(w, device=dev)
    step = _step_for(w, dev, window=37, window_mode=window_mode)
    step.pool(case["X"], 0, step.n_blk_max)
    args = (case["X"], case["K"], case["V"], case["Q"], case["q_idx"], case["w"],
            case["q_seq"], case["q_pos"], w.scale)
    step.run(*args)
    torch.cuda.synchronize()
    O_dev = step.O.clone()
    out = torch.empty(step.O.shape, dtype=torch.float32).pin_memory()
    step.set_output(out)
    step.run(*args)
    torch.cuda.synchronize()
    assert sfa.sfa_read_device_status(step.status) == 0
    assert torch.equal(out, O_dev.cpu())
    _check_queries(w, case, step, window=37)
