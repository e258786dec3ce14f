"""Seeded synthetic inputs for INT8-KV-cache attention.

This module is the one piece shared by the CUDA path's tests / benchmark and the CPU
oracle.  It only draws random numbers and lays out index arrays; it holds none of the
method's arithmetic (no quantisation, no attention).  bf16 values are produced as raw
16-bit patterns by round-to-nearest-even from fp32 draws.

Workloads (shapes and distributions of the pages' workloads; no public dataset is
involved, every input is synthetic):
  decode_1k      1 sequence, ctx 1024, 24 query / 4 KV heads, head_dim 256, Q/K/V ~ N(0,1)
                 bf16, contiguous pages (identity block table).
  decode_32k     1 sequence, ctx 32768, 24/4, head_dim 256, paged (block 16) with the block
                 table a random permutation, K elements multiplied by 8 with p = 0.01
                 (outliers), split-K with 512-key splits.
  prefill_32k    2048 new causal queries after 30720 history tokens (ctx 32768), 24/4,
                 head_dim 256, shuffled pages.
  decode_b64     64 sequences, ctx uniform in [512, 16384], 32 query / 8 KV heads,
                 head_dim 128, one pool of pages shuffled and dealt to the sequences; each
                 step also writes one new token per sequence.
  verify_32k     decode_32k's cache with 4 query rows per sequence (speculative / MTP verify):
                 the last 4 tokens of the sequence are the ones being verified, row i at
                 position ctx - 4 + i; each step rewrites those 4 tokens' K/V.
  sparse_32k     ctx 32768, 2048 queries at positions 30720..32767, 12 query heads on 1
                 KV head, head_dim 256, contiguous pages; query at position p attends to
                 sorted(2048 distinct positions uniform in [0, p-3] plus p-2, p-1, p).
"""
import numpy as np

SEED_BASE = 0x4B5651
BLOCK_SIZE = 16

CONFIGS = {
    "decode_1k": dict(kind="decode", index=0, batch=1, ctx=1024, hq=24, hkv=4, d=256,
                      paged="identity", k_outlier_p=0.0),
    "decode_32k": dict(kind="decode", index=1, batch=1, ctx=32768, hq=24, hkv=4, d=256,
                       paged="shuffled", k_outlier_p=0.01, split_rows=512),
    "prefill_32k": dict(kind="prefill", index=2, history=30720, chunk=2048, hq=24, hkv=4,
                        d=256, paged="shuffled", k_outlier_p=0.0),
    "decode_b64": dict(kind="decode", index=3, batch=64, ctx_range=(512, 16384), hq=32, hkv=8,
                       d=128, paged="shuffled", k_outlier_p=0.0),
    "verify_32k": dict(kind="decode", index=5, batch=1, ctx=32768, hq=24, hkv=4, d=256, nq=4,
                       paged="shuffled", k_outlier_p=0.01),
    "sparse_32k": dict(kind="sparse", index=4, ctx=32768, n_queries=2048, hq=12, hkv=1, d=256,
                       n_sample=2048, n_tail=3, paged="identity", k_outlier_p=0.0),
}


def f32_to_bf16_bits(x):
    """Round fp32 values to bf16 (nearest, ties to even); returns uint16 bit patterns."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    u = x.view(np.uint32).astype(np.uint64)
    rounded = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return rounded.astype(np.uint16)


def bf16_bits_to_f32(b):
    b = np.ascontiguousarray(b, dtype=np.uint16)
    return (b.astype(np.uint32) << 16).view(np.float32)


def normal_bf16(rng, shape, outlier_p=0.0, outlier_mul=8.0, chunk=1 << 24):
    """N(0,1) draws rounded to bf16.  With outlier_p > 0 each element is independently
    multiplied by outlier_mul with probability outlier_p (element-level outliers)."""
    n = int(np.prod(shape))
    out = np.empty(n, np.uint16)
    for s in range(0, n, chunk):
        e = min(n, s + chunk)
        x = rng.standard_normal(e - s, dtype=np.float32)
        if outlier_p > 0.0:
            hit = rng.random(e - s, dtype=np.float32) < outlier_p
            x[hit] *= outlier_mul
        out[s:e] = f32_to_bf16_bits(x)
    return out.reshape(shape)


def block_table(rng, ctx_lens, paged):
    """Per-sequence block tables over one pool of pages.  'identity' numbers pages in
    order; 'shuffled' deals a random permutation of the pool.  Rows are padded with -1
    past a sequence's last page.  Returns (table [n_seqs][max_blocks], num_blocks)."""
    ctx_lens = np.asarray(ctx_lens, np.int64)
    nb = (ctx_lens + BLOCK_SIZE - 1) // BLOCK_SIZE
    total = int(nb.sum())
    pool = np.arange(total, dtype=np.int32)
    if paged == "shuffled":
        pool = rng.permutation(total).astype(np.int32)
    table = np.full((len(ctx_lens), int(nb.max())), -1, np.int32)
    s = 0
    for i, n in enumerate(nb):
        table[i, :n] = pool[s:s + n]
        s += n
    return table, total


def sparse_cells(rng, positions, n_sample, n_tail):
    """Cell lists: for a query at position p, sorted(n_sample distinct positions drawn
    uniformly from [0, p - n_tail] plus the last n_tail positions p-n_tail+1 .. p)."""
    offsets = np.zeros(len(positions) + 1, np.int32)
    lists = []
    for i, p in enumerate(positions):
        low = p - n_tail + 1  # candidates for the uniform part are [0, low)
        k = min(n_sample, low)
        pick = rng.choice(low, size=k, replace=False) if k > 0 else np.zeros(0, np.int64)
        cells = np.concatenate([np.sort(pick), np.arange(low, p + 1)]).astype(np.int32)
        lists.append(cells)
        offsets[i + 1] = offsets[i] + len(cells)
    return offsets, np.concatenate(lists)


def make(name, seed=None, **override):
    """Build a workload dict for config `name` (overrides shrink it for tests)."""
    cfg = dict(CONFIGS[name])
    cfg.update(override)
    if seed is None:
        seed = SEED_BASE + cfg["index"]
    rng = np.random.default_rng(seed)
    kind, hq, hkv, d = cfg["kind"], cfg["hq"], cfg["hkv"], cfg["d"]
    w = dict(name=name, kind=kind, hq=hq, hkv=hkv, d=d, seed=seed, cfg=cfg,
             softmax_scale=1.0 / np.sqrt(d))
    if kind == "decode":
        B = cfg["batch"]
        if "ctx_range" in cfg:
            lo, hi = cfg["ctx_range"]
            ctx = rng.integers(lo, hi + 1, size=B).astype(np.int32)
        else:
            ctx = np.full(B, cfg["ctx"], np.int32)
        table, nblocks = block_table(rng, ctx, cfg["paged"])
        seq_idx = np.repeat(np.arange(B, dtype=np.int32), ctx)
        pos = np.concatenate([np.arange(c, dtype=np.int32) for c in ctx])
        w.update(batch=B, ctx_lens=ctx, max_ctx=int(ctx.max()), block_table=table,
                 num_blocks=nblocks, fill_seq=seq_idx, fill_pos=pos,
                 split_rows=cfg.get("split_rows", 512))
        w["k_fill"] = normal_bf16(rng, (len(pos), hkv, d), cfg["k_outlier_p"])
        w["v_fill"] = normal_bf16(rng, (len(pos), hkv, d))
        nq = cfg.get("nq", 1)
        w["nq"] = nq
        w["q"] = normal_bf16(rng, (B, hq, d) if nq == 1 else (B, nq, hq, d))
        # The step's new tokens of each sequence are its last nq positions; their K/V rows
        # are the ones already drawn for those positions, so writing them again leaves the
        # cache as generated and every step sees the same inputs.
        end = np.cumsum(ctx)
        rows = np.concatenate([np.arange(e - min(nq, c), e) for e, c in zip(end, ctx)]).astype(np.int64)
        w.update(new_seq=np.repeat(np.arange(B, dtype=np.int32), np.minimum(nq, ctx)),
                 new_pos=np.concatenate([np.arange(c - min(nq, c), c) for c in ctx]).astype(np.int32),
                 k_new=w["k_fill"][rows], v_new=w["v_fill"][rows])
    elif kind == "prefill":
        hist, T = cfg["history"], cfg["chunk"]
        ctx = hist + T
        table, nblocks = block_table(rng, [ctx], cfg["paged"])
        w.update(history=hist, n_tokens=T, ctx=ctx, block_table=table, num_blocks=nblocks,
                 fill_seq=np.zeros(ctx, np.int32), fill_pos=np.arange(ctx, dtype=np.int32))
        w["k_fill"] = normal_bf16(rng, (ctx, hkv, d), cfg["k_outlier_p"])
        w["v_fill"] = normal_bf16(rng, (ctx, hkv, d))
        w["q"] = normal_bf16(rng, (T, hq, d))
    elif kind == "sparse":
        ctx, N = cfg["ctx"], cfg["n_queries"]
        table, nblocks = block_table(rng, [ctx], cfg["paged"])
        positions = np.arange(ctx - N, ctx, dtype=np.int64)
        w.update(ctx=ctx, n_queries=N, block_table=table, num_blocks=nblocks,
                 positions=positions.astype(np.int32),
                 fill_seq=np.zeros(ctx, np.int32), fill_pos=np.arange(ctx, dtype=np.int32))
        w["k_fill"] = normal_bf16(rng, (ctx, hkv, d), cfg["k_outlier_p"])
        w["v_fill"] = normal_bf16(rng, (ctx, hkv, d))
        w["q"] = normal_bf16(rng, (N, hq, d))
        w["cell_offsets"], w["cells"] = sparse_cells(rng, positions, cfg["n_sample"],
                                                     cfg["n_tail"])
    else:
        raise ValueError(kind)
    return w
