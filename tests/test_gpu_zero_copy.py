"""The decode calls with their inputs and result in page-locked host memory (zero-copy).

On GB300 the GPU reads and writes page-locked host memory across the coherent host link, so a
decode step can take q, k_new, v_new and out straight from the host: no separate copy is
launched.  Gates: every output is bit-identical to the same call with device buffers, and the
cache bytes the fused step writes are too; pageable host memory is refused before any launch."""
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


def _host(bits):
    import torch
    return torch.from_numpy(np.ascontiguousarray(bits, dtype=np.uint16).view(np.int16)).view(torch.bfloat16).pin_memory()


def _same(a, b):
    return np.array_equal(np.asarray(a).view(np.uint32), np.asarray(b).view(np.uint32))


@pytest.mark.parametrize("route", [1, 2])
def test_decode_zero_copy_equals_device(kvq, route):
    w = W.make("decode_b64", seed=1400 + route, batch=3, ctx_range=(100, 2500), hq=24, hkv=4, d=256)
    cache, bt = gpu_cache_from(w, kvq)
    ctx = to_i32(w["ctx_lens"])
    qh = _host(w["q"])
    assert kvq.kvq_device_accessible(qh)
    dev = kvq.kvq_attn_decode_int8kv(cache, to_bf16_tensor(w["q"]), bt, ctx, w["max_ctx"], w["softmax_scale"],
                                     force_route=route).cpu().numpy()
    host = kvq.kvq_attn_decode_int8kv(cache, qh, bt, ctx, w["max_ctx"], w["softmax_scale"], force_route=route)
    assert host.device.type == "cpu" and host.is_pinned()
    import torch
    torch.cuda.synchronize()
    assert _same(host.numpy(), dev)
    assert kvq.kvq_device_status() == 0


def test_fused_step_and_verify_zero_copy(kvq):
    import torch
    w = W.make("decode_b64", seed=1410, batch=4, ctx_range=(50, 3000), hq=16, hkv=2, d=128, nq=3)
    B, nq, Hkv, D = w["batch"], w["nq"], w["hkv"], w["d"]
    kn = w["k_new"].reshape(B, nq, Hkv, D)
    vn = w["v_new"].reshape(B, nq, Hkv, D)
    ctx = to_i32(w["ctx_lens"])
    cache_d, bt = gpu_cache_from(w, kvq)
    cache_h, _ = gpu_cache_from(w, kvq)
    dev = kvq.kvq_decode_step_int8kv(cache_d, to_bf16_tensor(kn), to_bf16_tensor(vn), to_bf16_tensor(w["q"]), bt,
                                     ctx, w["max_ctx"], w["softmax_scale"]).cpu().numpy()
    out_h = torch.empty(dev.shape, dtype=torch.float32).pin_memory()
    kvq.kvq_decode_step_int8kv(cache_h, _host(kn), _host(vn), _host(w["q"]), bt, ctx, w["max_ctx"],
                               w["softmax_scale"], out=out_h)
    torch.cuda.synchronize()
    assert _same(out_h.numpy(), dev)
    for name in ("k", "v", "k_scale", "v_scale"):
        assert torch.equal(getattr(cache_d, name), getattr(cache_h, name)), name
    ver_d = kvq.kvq_attn_verify_int8kv(cache_d, to_bf16_tensor(w["q"]), bt, ctx, w["max_ctx"],
                                       w["softmax_scale"]).cpu().numpy()
    ver_h = kvq.kvq_attn_verify_int8kv(cache_h, _host(w["q"]), bt, ctx, w["max_ctx"], w["softmax_scale"])
    torch.cuda.synchronize()
    assert _same(ver_h.numpy(), ver_d)
    assert kvq.kvq_device_status() == 0


def test_pageable_host_memory_is_refused(kvq):
    import torch
    w = W.make("decode_b64", seed=1420, batch=2, ctx_range=(100, 300), hq=8, hkv=2, d=128)
    cache, bt = gpu_cache_from(w, kvq)
    q_pageable = torch.from_numpy(np.ascontiguousarray(w["q"]).view(np.int16)).view(torch.bfloat16)
    assert not kvq.kvq_device_accessible(q_pageable)
    with pytest.raises(ValueError):
        kvq.kvq_attn_decode_int8kv(cache, q_pageable, bt, to_i32(w["ctx_lens"]), w["max_ctx"], w["softmax_scale"])
    torch.cuda.synchronize()
    assert kvq.kvq_device_status() == 0


def test_host_cache_with_device_inputs_refused():
    """A cache left in host memory is refused before launch even when every other argument is a
    device tensor (the decode calls accept mapped host memory for q and out only)."""
    import torch

    import int8_kv_cache_quant_gb300 as kvq
    cache = kvq.KVCache(4, 1, 128, device="cpu")
    q = torch.zeros((1, 2, 128), dtype=torch.bfloat16, device="cuda")
    bt = torch.zeros((1, 4), dtype=torch.int32, device="cuda")
    ctx = torch.ones(1, dtype=torch.int32, device="cuda")
    with pytest.raises(ValueError):
        kvq.kvq_attn_decode_int8kv(cache, q, bt, ctx, 64, 0.1)
    rows = torch.zeros((1, 1, 128), dtype=torch.bfloat16, device="cuda")
    idx = torch.zeros(1, dtype=torch.int32, device="cuda")
    with pytest.raises(ValueError):
        kvq.kvq_quant_write(cache, rows, rows, idx, idx, bt)
