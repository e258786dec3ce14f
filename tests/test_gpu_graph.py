"""Every entry point of the hot path captured in a CUDA graph and replayed.

A decode step is launch-bound at short contexts, so a serving loop records it once and
replays it with new inputs copied into the captured buffers.  The library takes the
caller's stream, allocates nothing when it is given its output and workspace, and syncs
nowhere on the path, so each call can be captured.  Gates: the replay equals the eager call
bit for bit on the same inputs (every kernel of the path is deterministic: no atomics in
any sum), and a replay after new inputs are copied into the captured buffers equals the
eager call on those inputs."""
import numpy as np
import pytest

import workloads as W
from helpers import gpu_cache_from, to_bf16_tensor, to_i32

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def kvq():
    import int8_kv_cache_quant_gb300 as k
    k.lib()
    return k


def _capture(fn):
    """Run fn once eagerly on a side stream (first launches load the kernels), then record it
    into a graph."""
    import torch
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        fn()
    torch.cuda.current_stream().wait_stream(s)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fn()
    return g


def _same(a, b):
    return np.array_equal(a.view(np.uint32), b.view(np.uint32))


@pytest.mark.parametrize("route", [1, 2])
def test_decode_graph_replay(kvq, route):
    import torch
    w = W.make("decode_b64", seed=900 + route, batch=3, ctx_range=(200, 1400), hq=24, hkv=4, d=256)
    cache, bt = gpu_cache_from(w, kvq)
    q = to_bf16_tensor(w["q"])
    ctx = to_i32(w["ctx_lens"])
    out = torch.empty((w["batch"], w["hq"], w["d"]), dtype=torch.float32, device="cuda")
    ws = torch.empty(max(1, kvq.kvq_decode_workspace_bytes(w["batch"], w["hq"], w["max_ctx"], w["d"])),
                     dtype=torch.uint8, device="cuda")

    def call(o):
        kvq.kvq_attn_decode_int8kv(cache, q, bt, ctx, w["max_ctx"], w["softmax_scale"], out=o, workspace=ws,
                                   force_route=route, split_rows=256)

    g = _capture(lambda: call(out))
    out.zero_()
    g.replay()
    eager = torch.empty_like(out)
    call(eager)
    torch.cuda.synchronize()
    assert _same(out.cpu().numpy(), eager.cpu().numpy())
    # new query rows into the captured buffer, replay, against the eager call on them
    q.copy_(to_bf16_tensor(W.normal_bf16(np.random.default_rng(910 + route), tuple(q.shape))))
    g.replay()
    call(eager)
    torch.cuda.synchronize()
    assert _same(out.cpu().numpy(), eager.cpu().numpy())
    assert kvq.kvq_device_status() == 0


def test_fused_step_graph_replay(kvq):
    import torch
    w = W.make("decode_b64", seed=920, batch=4, ctx_range=(100, 2000), hq=32, hkv=8, d=128)
    cache, bt = gpu_cache_from(w, kvq)
    kn, vn, q = to_bf16_tensor(w["k_new"]), to_bf16_tensor(w["v_new"]), to_bf16_tensor(w["q"])
    ctx = to_i32(w["ctx_lens"])
    out = torch.empty((w["batch"], w["hq"], w["d"]), dtype=torch.float32, device="cuda")
    ws = torch.empty(max(1, kvq.kvq_verify_workspace_bytes(w["batch"], 1, w["hq"], w["max_ctx"], w["d"])),
                     dtype=torch.uint8, device="cuda")

    def call(o):
        kvq.kvq_decode_step_int8kv(cache, kn, vn, q, bt, ctx, w["max_ctx"], w["softmax_scale"], out=o,
                                   workspace=ws)

    k0, v0 = cache.k.clone(), cache.v.clone()
    g = _capture(lambda: call(out))
    for _ in range(3):  # the step rewrites the same rows: replays leave the cache as it was
        g.replay()
    eager = torch.empty_like(out)
    call(eager)
    torch.cuda.synchronize()
    assert _same(out.cpu().numpy(), eager.cpu().numpy())
    assert torch.equal(cache.k, k0) and torch.equal(cache.v, v0)
    assert kvq.kvq_device_status() == 0


def test_prefill_graph_replay(kvq):
    import torch
    # a shape whose units are split into two segments that meet through counters in the
    # workspace: every replay must start from zeroed counters
    w = W.make("prefill_32k", seed=930, history=2000, chunk=300, hq=12, hkv=2, d=256)
    cache, bt = gpu_cache_from(w, kvq)
    q = to_bf16_tensor(w["q"])
    T, Hq, D = w["n_tokens"], w["hq"], w["d"]
    out = torch.empty((T, Hq, D), dtype=torch.float32, device="cuda")
    ws = torch.empty(kvq.kvq_prefill_workspace_bytes(T, Hq, w["hkv"], w["history"], D), dtype=torch.uint8,
                     device="cuda")

    def call(o):
        kvq.kvq_attn_prefill_int8(cache, q, w["history"], bt[0], w["softmax_scale"], out=o, workspace=ws)

    assert kvq.kvq_prefill_split_tiles(T, Hq, w["history"], torch.cuda.get_device_properties(0).multi_processor_count) > 0

    g = _capture(lambda: call(out))
    for _ in range(2):
        out.zero_()
        g.replay()
    eager = torch.empty_like(out)
    call(eager)
    torch.cuda.synchronize()
    assert _same(out.cpu().numpy(), eager.cpu().numpy())
    assert kvq.kvq_device_status() == 0


def test_sparse_graph_replay(kvq):
    import torch
    w = W.make("sparse_32k", seed=940, ctx=900, n_queries=40, n_sample=300)
    cache, bt = gpu_cache_from(w, kvq)
    q = to_bf16_tensor(w["q"])
    offs, cells = to_i32(w["cell_offsets"]), to_i32(w["cells"])
    N, Hq, D = w["n_queries"], w["hq"], w["d"]
    out = torch.empty((N, Hq, D), dtype=torch.float32, device="cuda")
    ws = torch.empty(kvq.kvq_sparse_workspace_bytes(int(bt.shape[1]), w["hkv"], D), dtype=torch.uint8,
                     device="cuda")

    def call(o):
        kvq.kvq_attn_sparse_int8kv(cache, q, offs, cells, bt[0], w["softmax_scale"], out=o, workspace=ws)

    g = _capture(lambda: call(out))
    out.zero_()
    g.replay()
    eager = torch.empty_like(out)
    call(eager)
    torch.cuda.synchronize()
    assert _same(out.cpu().numpy(), eager.cpu().numpy())
    assert kvq.kvq_device_status() == 0
