"""The bench's algorithmic work per step (CPU): closed forms of the bytes each stage must move,
for the bf16 and the q8_0 caches."""
import importlib
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _bench():
    import __graft_entry__
    __graft_entry__.build()
    sys.path.insert(0, ROOT)
    return importlib.import_module("bench")


def test_gathered_bytes_per_cell():
    b = _bench()
    import indexer_selected_sparse_block_gb300 as sfa
    w = sfa.WORKLOADS["decode_32x131072"]          # 576-wide K, V = K, one KV head
    att = [512 * 4 + 1] * w.n_q                      # 512 kept blocks of 4 cells + a 1-cell tail
    assert b.algorithmic(w, att)["gathered_kv_bytes"] == 32 * 2049 * 1152
    assert b.algorithmic(w, att, kv="q8_0")["gathered_kv_bytes"] == 32 * 2049 * 624
    v = sfa.WORKLOADS["decode_4x1048576"]           # 512-wide K and separate V, two KV heads
    att = [256 * 8 + 1] * v.n_q
    assert b.algorithmic(v, att)["gathered_kv_bytes"] == 4 * 2049 * 2 * (512 + 512) * 2
    assert b.algorithmic(v, att, kv="q8_0")["gathered_kv_bytes"] == 4 * 2049 * 2 * (544 + 544)
    # the attention's flops do not depend on the cache type
    assert b.algorithmic(v, att)["attend_flops"] == b.algorithmic(v, att, kv="q8_0")["attend_flops"]


def test_pooled_key_bytes():
    b = _bench()
    import indexer_selected_sparse_block_gb300 as sfa
    w = sfa.WORKLOADS["decode_32x131072"]
    a = b.algorithmic(w, [1] * w.n_q, bounded=True)
    nb = (w.depth + 1) // w.compress_ratio
    assert a["kbar_bytes"] == w.n_q * nb * (2 * w.d_idx + 4)     # hi halves + bound factor
    assert a["score_bytes"] == w.n_q * nb * 8                     # lower + upper bounds
    e = b.algorithmic(w, [1] * w.n_q, bounded=False)
    assert e["kbar_bytes"] == w.n_q * nb * 4 * w.d_idx             # hi + lo halves
    c = b.algorithmic(w, [1] * w.n_q, bounded="i8")
    assert c["kbar_bytes"] == w.n_q * nb * (w.d_idx + 8)           # codes + scale, bound factor
    assert c["score_bytes"] == a["score_bytes"]


def test_conflicting_selection_flags_are_refused():
    """--exact and --bounded together stop at argument parsing, before any device work."""
    import subprocess
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--exact", "--bounded"],
                       capture_output=True, text=True, cwd=ROOT, timeout=300)
    assert r.returncode == 2
    assert "--exact and --bounded exclude each other" in r.stderr


def test_traffic_records_name_existing_kernels():
    """Each DRAM-traffic record the bench can report names a workload the bench knows, a source
    file that defines the kernel it was taken on, and read + write bytes that add up."""
    import json
    import indexer_selected_sparse_block_gb300 as sfa
    with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
        records = json.load(f)
    assert records
    csrc = os.path.join(ROOT, "indexer_selected_sparse_block_gb300", "csrc")
    for key, rec in records.items():
        stage, workload = key.split("@")
        assert stage in ("scores", "topk", "attend"), key
        assert workload in sfa.WORKLOADS, key
        with open(os.path.join(csrc, rec["source"])) as f:
            src = f.read()
        assert rec["kernel"].split("<")[0] in src, key
        assert rec["dram_bytes_per_launch"] == rec["dram_read"] + rec["dram_write"], key
        assert len(rec["src_sha256_16"]) == 16 and rec["command"].startswith("ncu "), key
