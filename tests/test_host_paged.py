"""Host logic of the paged cell layout (CPU): the seeded page table, the scatter into cells,
and the step runner's checks of its paged arguments."""
import pytest
import torch

from indexer_selected_sparse_block_gb300.inputs import make_cell_map, to_cells


@pytest.mark.parametrize("n_seq,n_pos,page,spare", [(3, 130, 16, 2), (1, 64, 64, 0), (4, 1, 8, 5)])
def test_cell_map_is_a_shuffled_page_table(n_seq, n_pos, page, spare):
    cell_of, n_cells = make_cell_map(n_seq, n_pos, page=page, spare_pages=spare, seed=11)
    pps = -(-n_pos // page)
    assert cell_of.dtype == torch.int32 and tuple(cell_of.shape) == (n_seq, n_pos)
    assert n_cells == (n_seq * pps + spare) * page
    flat = cell_of.reshape(-1).long()
    assert flat.min() >= 0 and flat.max() < n_cells
    assert torch.unique(flat).numel() == flat.numel()               # no cell holds two positions
    # positions fill whole pages in order: the cell of t is page(t // page) * page + t % page
    t = torch.arange(n_pos)
    off = cell_of.long() - (t % page)[None, :]
    assert torch.all(off % page == 0)
    pages = off // page
    assert torch.all(pages[:, t] == pages[:, (t // page) * page])
    assert len(set(pages[:, ::page].reshape(-1).tolist())) == n_seq * pps
    again, _ = make_cell_map(n_seq, n_pos, page=page, spare_pages=spare, seed=11)
    assert torch.equal(cell_of, again)                               # seeded


def test_cell_map_seed_changes_the_table():
    a, _ = make_cell_map(4, 256, page=16, spare_pages=4, seed=1)
    b, _ = make_cell_map(4, 256, page=16, spare_pages=4, seed=2)
    assert not torch.equal(a, b)


def test_to_cells_places_every_row_in_its_cell():
    cell_of, n_cells = make_cell_map(3, 70, page=8, spare_pages=3, seed=5)
    x = torch.randn(3, 70, 2, 5)
    cells = to_cells(x, cell_of, n_cells)
    assert tuple(cells.shape) == (n_cells, 2, 5)
    for s in range(3):
        assert torch.equal(cells[cell_of[s].long()], x[s])
    used = torch.zeros(n_cells, dtype=torch.bool)
    used[cell_of.reshape(-1).long()] = True
    assert torch.all(cells[~used] == 0)


def _step(**kw):
    import __graft_entry__
    __graft_entry__.build()
    import indexer_selected_sparse_block_gb300 as sfa
    args = dict(n_seq=2, n_tok_cap=64, n_q=2, h_q=16, h_kv=1, dkq=576, dv=512, h_idx=4, d_idx=64,
                compress_ratio=4, indexer_top_k=4, n_blk_max=16, device="cpu")
    args.update(kw)
    return sfa.SfaStep(**args)


def test_step_checks_its_cell_map():
    with pytest.raises(ValueError):
        _step(cell_of=torch.zeros((2, 63), dtype=torch.int32))      # wrong shape
    with pytest.raises(ValueError):
        _step(cell_of=torch.zeros((2, 64), dtype=torch.int64))      # wrong dtype
    with pytest.raises(ValueError):
        _step(cell_of=torch.zeros((2, 64), dtype=torch.int32), key_transform={"norm": 1})
    st = _step(cell_of=torch.zeros((2, 64), dtype=torch.int32))
    assert st.cell_of is not None and not st.dense
