"""kvq_attn_sparse_int8kv on the GPU against the oracle (FP64 Part A over the cell lists).
Gate: 2e-3 normalised max-abs error; the FP32 design lands near 1e-6 (DESIGN_TOL 1e-4)."""
import numpy as np
import pytest

import workloads as W
from helpers import gpu_cache_from, host_cache_from, norm_max_err, sample_units, to_bf16_tensor, to_i32

pytestmark = pytest.mark.gpu

GATE = 2e-3
DESIGN_TOL = 1e-4


@pytest.fixture(scope="module")
def kvq():
    import int8_kv_cache_quant_gb300 as k
    k.lib()
    return k


def _sparse(kvq, w, cache, offsets, cells):
    out = kvq.kvq_attn_sparse_int8kv(cache, to_bf16_tensor(w["q"]), to_i32(offsets), to_i32(cells),
                                     to_i32(w["block_table"][0]), w["softmax_scale"])
    return out.cpu().numpy()


@pytest.mark.parametrize("d,hq,hkv", [(256, 12, 1), (128, 8, 2), (256, 4, 4)])
def test_small_random_cells(kvq, oracle, d, hq, hkv):
    w = W.make("sparse_32k", seed=500 + hq, ctx=700, n_queries=37, n_sample=150, hq=hq, hkv=hkv, d=d)
    cache, _ = gpu_cache_from(w, kvq)
    got = _sparse(kvq, w, cache, w["cell_offsets"], w["cells"])
    hc = host_cache_from(w, oracle)
    ref = oracle.sparse_f64(hc, w["q"], w["cell_offsets"], w["cells"], w["block_table"][0], w["softmax_scale"])
    assert norm_max_err(got, ref) <= DESIGN_TOL
    assert kvq.kvq_device_status() == 0


def test_every_cell_equals_causal_and_edge_lists(kvq, oracle):
    # ctx 300, 20 queries at 280..299 reading every cell of their causal prefix (the
    # page's "every cell" case); plus an empty list and a single cell.
    w = W.make("sparse_32k", seed=510, ctx=300, n_queries=20, n_sample=10, hq=12, hkv=1, d=256)
    pos = w["positions"]
    lists = [np.arange(p + 1, dtype=np.int32) for p in pos]
    lists[3] = np.zeros(0, np.int32)
    lists[4] = np.array([17], np.int32)
    offsets = np.concatenate([[0], np.cumsum([len(x) for x in lists])]).astype(np.int32)
    cells = np.concatenate(lists).astype(np.int32)
    cache, _ = gpu_cache_from(w, kvq)
    got = _sparse(kvq, w, cache, offsets, cells)
    assert not got[3].any()
    hc = host_cache_from(w, oracle)
    ref = oracle.sparse_f64(hc, w["q"], offsets, cells, w["block_table"][0], w["softmax_scale"])
    assert norm_max_err(got, ref) <= DESIGN_TOL


def test_sparse_32k_full_sampled(kvq, oracle):
    """Workload sparse_32k at full size (ctx 32768, 2048 queries x 2051 cells, 12 q heads per
    KV head, head_dim 256): sampled (query, head) outputs against FP64."""
    w = W.make("sparse_32k")
    cache, _ = gpu_cache_from(w, kvq)
    got = _sparse(kvq, w, cache, w["cell_offsets"], w["cells"])
    hc = host_cache_from(w, oracle)
    units = sample_units(w["n_queries"], w["hq"], 256, seed=11)
    ref = oracle.sparse_f64(hc, w["q"], w["cell_offsets"], w["cells"], w["block_table"][0],
                            w["softmax_scale"], units=units)
    err = norm_max_err(got.reshape(-1, w["d"])[units], ref)
    print("sparse_32k normalised max err (sampled)", err)
    assert err <= GATE and err <= DESIGN_TOL
