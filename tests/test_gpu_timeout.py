"""The failure path of the bounded waits, made to run on purpose without faulting the GPU.

kvq_debug_fault_inject makes one CTA leave one copy un-issued (nothing is left in flight: its
barrier simply never completes) and shortens every wait to about a millisecond.  The consumer's
wait must run out, the kernel must report KVQ_DEV_TIMEOUT through the status word, wait (bounded)
for the copies it did issue, drop that CTA's result and return; the device stays usable, and the
next call with the injection off is correct.
"""
import numpy as np
import pytest

import workloads as W
from helpers import gpu_cache_from, host_cache_from, norm_max_err, to_bf16_tensor, to_i32

pytestmark = pytest.mark.gpu

BUDGET = 2_000_000  # SM clock cycles, about 1 ms


@pytest.fixture(scope="module")
def kvq():
    import int8_kv_cache_quant_gb300 as k
    k.lib()
    return k


def _run_injected(kvq, mode, fn):
    kvq.kvq_device_status()  # clear earlier bits
    kvq.kvq_debug_fault_inject(mode, BUDGET)
    try:
        out = fn()
        st = kvq.kvq_device_status()
    finally:
        kvq.kvq_debug_fault_inject(0, 0)
    return out, st


def test_decode_wait_runs_out_and_the_device_recovers(kvq, oracle):
    w = W.make("decode_32k", seed=1701, batch=2, ctx=900, hq=24, hkv=4, d=256)
    cache, bt = gpu_cache_from(w, kvq)
    hc = host_cache_from(w, oracle)
    ref = oracle.decode_f64(hc, w["q"], w["block_table"], w["ctx_lens"], w["softmax_scale"])
    q, ctx = to_bf16_tensor(w["q"]), to_i32(w["ctx_lens"])
    G = w["hq"] // w["hkv"]

    def call(route):
        return kvq.kvq_attn_decode_int8kv(cache, q, bt, ctx, w["max_ctx"], w["softmax_scale"], force_route=route,
                                          split_rows=256)

    # single route: CTA 0 is (sequence 0, KV head 0); its rows come out as zeros
    out, st = _run_injected(kvq, 1, lambda: call(1).cpu().numpy())
    assert st & kvq.kvq.DEV_TIMEOUT, st
    assert np.all(out[0, :G] == 0)
    assert norm_max_err(out[0, G:], ref[0, G:]) <= 1e-4
    assert norm_max_err(out[1], ref[1]) <= 1e-4
    # split route: CTA 0 is split 0 of (sequence 0, KV head 0); its partial is dropped, the
    # merge combines the others
    out, st = _run_injected(kvq, 1, lambda: call(2).cpu().numpy())
    assert st & kvq.kvq.DEV_TIMEOUT, st
    assert np.isfinite(out).all()
    assert norm_max_err(out[0, G:], ref[0, G:]) <= 1e-4 and norm_max_err(out[1], ref[1]) <= 1e-4
    assert norm_max_err(out[0, :G], ref[0, :G]) > 1e-3  # the first 256 keys are missing
    # the next calls, injection off: correct, no status bits
    for route in (1, 2):
        got = call(route).cpu().numpy()
        assert norm_max_err(got, ref) <= 1e-4
    assert kvq.kvq_device_status() == 0


def test_prefill_wait_runs_out_and_the_device_recovers(kvq, oracle):
    import torch
    w = W.make("prefill_32k", seed=1702, history=100, chunk=200, hq=6, hkv=1, d=256)
    cache, bt = gpu_cache_from(w, kvq)
    hc = host_cache_from(w, oracle)
    emul = oracle.prefill_int8_emul(hc, w["q"], w["history"], w["block_table"][0], w["softmax_scale"])
    q = to_bf16_tensor(w["q"])
    T, Hq, D = w["n_tokens"], w["hq"], w["d"]

    def call():
        out = torch.full((T, Hq, D), 7.0, dtype=torch.float32, device="cuda")
        kvq.kvq_attn_prefill_int8(cache, q, w["history"], bt[0], w["softmax_scale"], out=out)
        return out.cpu().numpy()

    # attention CTA 0 is the last query tile (rows 128..199) of query head 0: left unwritten
    out, st = _run_injected(kvq, 2, call)
    assert st & kvq.kvq.DEV_TIMEOUT, st
    assert np.all(out[128:, 0] == 7.0)
    mask = np.ones((T, Hq), bool)
    mask[128:, 0] = False
    assert norm_max_err(out[mask], emul[mask]) <= 1e-4
    got = call()
    assert norm_max_err(got, emul) <= 1e-4
    assert kvq.kvq_device_status() == 0


def test_fault_inject_rejects_unknown_modes(kvq):
    with pytest.raises(kvq.KvqError):
        kvq.kvq_debug_fault_inject(7, 0)


def test_sparse_wait_runs_out_and_the_device_recovers(kvq, oracle):
    w = W.make("sparse_32k", seed=1703, ctx=640, n_queries=6, hq=4, hkv=1, d=128, n_sample=300)
    cache, bt = gpu_cache_from(w, kvq)
    hc = host_cache_from(w, oracle)
    ref = oracle.sparse_f64(hc, w["q"], w["cell_offsets"], w["cells"], w["block_table"][0], w["softmax_scale"])
    q, off, cells, row = to_bf16_tensor(w["q"]), to_i32(w["cell_offsets"]), to_i32(w["cells"]), to_i32(w["block_table"][0])
    assert int(w["cell_offsets"][1]) > 64  # query 0 has a second chunk

    def call():
        return kvq.kvq_attn_sparse_int8kv(cache, q, off, cells, row, w["softmax_scale"]).cpu().numpy()

    # the CTA of (query 0, KV head 0) leaves its second chunk un-issued: its rows are zeros
    out, st = _run_injected(kvq, 3, call)
    assert st & kvq.kvq.DEV_TIMEOUT, st
    assert np.all(out[0] == 0)
    assert norm_max_err(out[1:], ref[1:]) <= 1e-4
    got = call()
    assert norm_max_err(got, ref) <= 1e-4
    assert kvq.kvq_device_status() == 0
