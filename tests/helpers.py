"""Shared helpers of the GPU tests: upload seeded workloads, fill the caches on both sides
(the GPU cache by the CUDA path, the host cache by the oracle), and the error metric."""
import numpy as np

import workloads as W


def to_bf16_tensor(bits, device="cuda"):
    import torch
    a = np.ascontiguousarray(bits, dtype=np.uint16).view(np.int16)
    return torch.from_numpy(a).to(device).view(torch.bfloat16)


def to_i32(a, device="cuda"):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).to(device)


def gpu_cache_from(w, kvq, chunk_tokens=1 << 16):
    """Build a device cache and fill it with the workload's tokens through kvq_quant_write."""
    cache = kvq.KVCache(w["num_blocks"], w["hkv"], w["d"])
    bt = to_i32(w["block_table"])
    n = len(w["fill_pos"])
    for s in range(0, n, chunk_tokens):
        e = min(n, s + chunk_tokens)
        kvq.kvq_quant_write(cache, to_bf16_tensor(w["k_fill"][s:e]), to_bf16_tensor(w["v_fill"][s:e]),
                            to_i32(w["fill_seq"][s:e]), to_i32(w["fill_pos"][s:e]), bt)
    return cache, bt


def host_cache_from(w, oracle):
    """Build the oracle's host cache from the same tokens through the oracle's quantiser."""
    c = oracle.HostCache(w["num_blocks"], w["hkv"], w["d"])
    skipped = oracle.kv_quant_write(c, w["k_fill"], w["v_fill"], w["fill_seq"], w["fill_pos"],
                                    w["block_table"])
    assert skipped == 0
    return c


def norm_max_err(got, ref):
    """max |got - ref| / RMS(ref): the acceptance metric of the outputs."""
    ref = np.asarray(ref, np.float64)
    got = np.asarray(got, np.float64)
    rms = np.sqrt(np.mean(ref ** 2))
    return float(np.max(np.abs(got - ref)) / rms) if rms > 0 else float(np.max(np.abs(got - ref)))


def sample_units(n_rows, n_heads, k, seed):
    """k distinct (row, head) unit ids, always including the first and last rows."""
    rng = np.random.default_rng(seed)
    total = n_rows * n_heads
    k = min(k, total)
    pick = set(rng.choice(total, size=k, replace=False).tolist())
    pick.update([0, total - 1])
    return np.array(sorted(pick), np.int64)
