"""Seeded synthetic workloads for paged top-k sparse MLA.

This module only draws inputs: shapes, block tables, lengths, prefix trees and
random values.  It contains none of the method's arithmetic, so both the CUDA
library and the CPU oracle can be fed from it.

The synthetic data stands in for the agentic traces that the sources measure
on (median 142K-token inputs, >96% prefix reuse, subagents forking from a
parent context, MTP3 decode, chunked prefill on a cached prefix):

* bf16 q, q_pe, latent and rope values ~ N(0, 1);
* indexer q and k are integers in [-r, r] (r = 8, or 4 for the tiny shape),
  stored as E4M3 (exact for such integers);
* indexer head weights drawn uniformly from {0.25, 0.5, 1};
* indexer key scales 1.0 (tests also use powers of two);
* physical block ids are a random permutation of the pool;
* with FP4 indexer keys (``key_format="e2m1"``), every key element is a
  uniformly drawn 4-bit E2M1 code (all sixteen, so the values 0, +-0.5, +-1,
  +-1.5, +-2, +-3, +-4, +-6), two codes packed per byte, low nibble first.

Five named shapes (``make_config(i)``):
  1 tiny decode: 2 seqs x 1 query, ctx 256, bs 16, 8 shared prefix blocks,
    pool of 32 blocks; 8 heads, latent 64 + rope 16, indexer 4 x 32, top-k 64.
  2 decode: 32 seqs x 1 query, ctx ~ U[8192, 32768], bs 64; 64 heads,
    latent 512 (+4 fp32 scales) + rope 64, indexer 64 x 128, top-k 2048.
  3 agentic MTP decode: 64 seqs x 4 queries; ctx lognormal(median 142K,
    sigma 0.6) clipped to [16K, 256K]; 13 parents with forked children
    (1 + Poisson(3) each) sharing >= 96% of their blocks.
  4 long-context decode: 8 seqs x 1 query, ctx 1,048,576.
  5 chunked prefill: 1 seq, 131,072 cached + 8,192 new query tokens.
``make_config(i, key_format="e2m1")`` gives shapes 2-5 with FP4 indexer keys.
"""

from dataclasses import dataclass, field, replace
import math

import numpy as np
import torch


@dataclass(frozen=True)
class Dims:
    n_heads: int = 64
    d_latent: int = 512
    d_rope: int = 64
    quant_tile: int = 128
    n_idx_heads: int = 64
    d_index: int = 128
    top_k: int = 2048
    block_size: int = 64
    n_layers: int = 1
    idx_range: int = 8
    key_format: str = "e4m3"   # indexer keys: "e4m3" (one byte per element) or "e2m1" (packed FP4)

    @property
    def softmax_scale(self) -> float:
        return 1.0 / math.sqrt(self.d_latent + self.d_rope)

    @property
    def key_bytes(self) -> int:
        return self.d_index if self.key_format == "e4m3" else self.d_index // 2


TINY = Dims(n_heads=8, d_latent=64, d_rope=16, quant_tile=64, n_idx_heads=4, d_index=32,
            top_k=64, block_size=16, idx_range=4)
FULL = Dims()


@dataclass
class Workload:
    name: str
    dims: Dims
    num_blocks: int
    block_table: torch.Tensor        # int32 [B, max_blocks], -1 beyond each sequence
    seq_lens: torch.Tensor           # int32 [B], includes this step's tokens
    query_start_loc: torch.Tensor    # int32 [B + 1]
    slot_mapping: torch.Tensor       # int64 [T], slots of this step's tokens
    cached_slots: torch.Tensor       # int64 [Nc], slots holding earlier tokens (deduplicated)
    slot_latent: torch.Tensor        # bf16 [num_blocks * bs, D_L]: value of each physical slot
    slot_rope: torch.Tensor          # bf16 [num_blocks * bs, D_R]
    slot_idx_k: torch.Tensor         # uint8 [num_blocks * bs, key_bytes] (E4M3, or packed E2M1)
    slot_idx_s: torch.Tensor         # fp32 [num_blocks * bs]
    new_latent: torch.Tensor         # bf16 [T, D_L]
    new_rope: torch.Tensor           # bf16 [T, D_R]
    new_idx_k: torch.Tensor          # uint8 [T, key_bytes]
    new_idx_s: torch.Tensor          # fp32 [T]
    q: torch.Tensor                  # bf16 [T, H, D_L]
    q_pe: torch.Tensor               # bf16 [T, H, D_R]
    q_idx: torch.Tensor              # uint8 [T, H_I, D_I]
    w: torch.Tensor                  # fp32 [T, H_I]
    max_q: int
    max_ctx: int
    parents: list = field(default_factory=list)

    @property
    def batch(self) -> int:
        return int(self.seq_lens.numel())

    @property
    def n_tokens(self) -> int:
        return int(self.slot_mapping.numel())


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def _int_e4m3(shape, r: int, g, device) -> torch.Tensor:
    v = torch.randint(-r, r + 1, shape, generator=g, device=device, dtype=torch.int32)
    return v.to(torch.float32).to(torch.float8_e4m3fn).view(torch.uint8)


def _packed_e2m1(shape, g, device) -> torch.Tensor:
    """Uniform 4-bit codes, two per byte: [..., D] elements -> [..., D/2] bytes."""
    *lead, d = shape
    return torch.randint(0, 256, (*lead, d // 2), generator=g, device=device, dtype=torch.int32).to(torch.uint8)


def _keys(shape, dims, g, device) -> torch.Tensor:
    if dims.key_format == "e2m1":
        return _packed_e2m1(shape, g, device)
    return _int_e4m3(shape, dims.idx_range, g, device)


def _normal_bf16(shape, g, device) -> torch.Tensor:
    return torch.randn(shape, generator=g, device=device, dtype=torch.float32).to(torch.bfloat16)


def build_workload(name: str, dims: Dims, ctx_lens, n_q, *, seed: int, device="cpu",
                   share=None, slack_blocks: int = 0, idx_scale=None) -> Workload:
    """Draw a workload.

    ctx_lens[b]: total tokens of sequence b after this step (cached + new);
    n_q[b]: new query tokens of sequence b this step (its last positions);
    share[b] = (parent, n_blocks): sequence b's first n_blocks logical blocks
    are the parent's physical blocks (parent must come earlier).
    """
    rng = np.random.default_rng(seed)
    bs = dims.block_size
    ctx_lens = [int(c) for c in ctx_lens]
    n_q = [int(x) for x in n_q]
    b_count = len(ctx_lens)
    share = share or [(-1, 0)] * b_count
    nblk = [(c + bs - 1) // bs for c in ctx_lens]
    private = [nblk[b] - share[b][1] for b in range(b_count)]
    num_blocks = sum(private) + slack_blocks
    perm = rng.permutation(num_blocks).astype(np.int64)
    max_blocks = max(nblk)
    bt = np.full((b_count, max_blocks), -1, dtype=np.int64)
    nxt = 0
    for b in range(b_count):
        par, ns = share[b]
        if par >= 0:
            assert par < b and ns <= nblk[par]
            bt[b, :ns] = bt[par, :ns]
        bt[b, ns:nblk[b]] = perm[nxt:nxt + private[b]]
        nxt += private[b]
    # slots of this step's tokens (the last n_q positions of each sequence)
    slot_map, cached = [], set()
    for b in range(b_count):
        pos_new = np.arange(ctx_lens[b] - n_q[b], ctx_lens[b], dtype=np.int64)
        slot_map.append(bt[b, pos_new // bs] * bs + pos_new % bs)
    slot_map = np.concatenate(slot_map) if slot_map else np.zeros(0, np.int64)
    cached_slots = []
    for b in range(b_count):
        n_c = ctx_lens[b] - n_q[b]
        pos = np.arange(n_c, dtype=np.int64)
        cached_slots.append(bt[b, pos // bs] * bs + pos % bs)
    cached_slots = np.unique(np.concatenate(cached_slots)) if cached_slots else np.zeros(0, np.int64)
    assert not np.isin(slot_map, cached_slots).any(), "a new token would overwrite a cached slot"
    qsl = np.concatenate([[0], np.cumsum(n_q)]).astype(np.int64)

    g = _gen(seed, device)
    n_slots = num_blocks * bs
    t = int(qsl[-1])
    r = dims.idx_range
    d = dims
    slot_latent = _normal_bf16((n_slots, d.d_latent), g, device)
    slot_rope = _normal_bf16((n_slots, d.d_rope), g, device)
    slot_idx_k = _keys((n_slots, d.d_index), d, g, device)
    new_latent = _normal_bf16((t, d.d_latent), g, device)
    new_rope = _normal_bf16((t, d.d_rope), g, device)
    new_idx_k = _keys((t, d.d_index), d, g, device)
    q = _normal_bf16((t, d.n_heads, d.d_latent), g, device)
    q_pe = _normal_bf16((t, d.n_heads, d.d_rope), g, device)
    q_idx = _int_e4m3((t, d.n_idx_heads, d.d_index), r, g, device)
    wsel = torch.randint(0, 3, (t, d.n_idx_heads), generator=g, device=device)
    w = torch.tensor([0.25, 0.5, 1.0], device=device, dtype=torch.float32)[wsel]
    if idx_scale is None:
        slot_idx_s = torch.ones(n_slots, device=device, dtype=torch.float32)
        new_idx_s = torch.ones(t, device=device, dtype=torch.float32)
    else:
        vals = torch.tensor(idx_scale, device=device, dtype=torch.float32)
        slot_idx_s = vals[torch.randint(0, len(idx_scale), (n_slots,), generator=g, device=device)]
        new_idx_s = vals[torch.randint(0, len(idx_scale), (t,), generator=g, device=device)]

    as_t = lambda a, dt: torch.as_tensor(a, dtype=dt).to(device)
    return Workload(
        name=name, dims=dims, num_blocks=num_blocks,
        block_table=as_t(bt, torch.int32), seq_lens=as_t(ctx_lens, torch.int32),
        query_start_loc=as_t(qsl, torch.int32), slot_mapping=as_t(slot_map, torch.int64),
        cached_slots=as_t(cached_slots, torch.int64),
        slot_latent=slot_latent, slot_rope=slot_rope, slot_idx_k=slot_idx_k, slot_idx_s=slot_idx_s,
        new_latent=new_latent, new_rope=new_rope, new_idx_k=new_idx_k, new_idx_s=new_idx_s,
        q=q, q_pe=q_pe, q_idx=q_idx, w=w, max_q=max(n_q) if n_q else 0,
        max_ctx=max(ctx_lens) if ctx_lens else 0, parents=[s[0] for s in share])


def agentic_tree(seed: int, n_seqs: int = 64, n_parents: int = 13, n_q: int = 4,
                 median: float = 142_000.0, sigma: float = 0.6, lo: int = 16_384, hi: int = 262_144,
                 block_size: int = 64, ctx_scale: float = 1.0):
    """Context lengths and prefix sharing of an agentic batch.

    Parents draw lengths from lognormal(ln median, sigma) clipped to [lo, hi];
    each parent gets 1 + Poisson(3) forked children (adjusted so the batch has
    n_seqs sequences); a child is g ~ U[1.0, 1.04] times its parent's length and
    shares floor(f * L_child / bs) of the parent's blocks, f ~ U[0.96, 1.0],
    never a block that holds either sequence's new tokens.  ``ctx_scale``
    shrinks every length (for small test cases).
    """
    rng = np.random.default_rng(seed + 1000)
    kids = 1 + rng.poisson(3.0, size=n_parents)
    want = n_seqs - n_parents
    while kids.sum() > want:
        i = rng.integers(n_parents)
        if kids[i] > 1:
            kids[i] -= 1
    while kids.sum() < want:
        kids[rng.integers(n_parents)] += 1
    lens, share = [], []
    for pidx in range(n_parents):
        lp = int(np.clip(rng.lognormal(math.log(median), sigma), lo, hi) * ctx_scale)
        lp = max(lp, n_q + 1)
        parent_row = len(lens)
        lens.append(lp)
        share.append((-1, 0))
        for _ in range(int(kids[pidx])):
            lc = max(int(lp * rng.uniform(1.0, 1.04)), n_q + 1)
            f = rng.uniform(0.96, 1.0)
            ns = min(int(f * lc) // block_size, (lp - n_q) // block_size, (lc - n_q) // block_size)
            lens.append(lc)
            share.append((parent_row, max(ns, 0)))
    return lens, share


def make_config(i: int, device="cpu", *, scale: float = 1.0, key_format: str = "e4m3") -> Workload:
    """The five named shapes; ``scale`` < 1 shrinks context lengths (tests only); ``key_format="e2m1"``
    draws FP4 indexer keys for shapes 2-5 (names get a "-fp4keys" suffix)."""
    if key_format not in ("e4m3", "e2m1"):
        raise ValueError(f"unknown key format {key_format!r}")
    if key_format == "e2m1" and i == 1:
        raise ValueError("FP4 indexer keys are built for the 128-dim indexer of shapes 2-5")
    full = FULL if key_format == "e4m3" else replace(FULL, key_format=key_format)
    sfx = "" if key_format == "e4m3" else "-fp4keys"
    if i == 1:
        share = [(-1, 0), (0, 8)]
        return build_workload("tiny-decode", TINY, [256, 256], [1, 1], seed=0, device=device,
                              share=share, slack_blocks=8)
    if i == 2:
        rng = np.random.default_rng(1)
        lens = rng.integers(8192, 32768 + 1, size=32)
        lens = np.maximum((lens * scale).astype(np.int64), 2)
        return build_workload("decode-b32-ctx8k-32k" + sfx, full, lens, [1] * 32, seed=1, device=device)
    if i == 3:
        lens, share = agentic_tree(2, ctx_scale=scale)
        return build_workload("agentic-mtp4-b64-ctx142k" + sfx, full, lens, [4] * len(lens), seed=2,
                              device=device, share=share)
    if i == 4:
        n = max(int(1_048_576 * scale), 2)
        return build_workload("longctx-b8-ctx1m" + sfx, full, [n] * 8, [1] * 8, seed=3, device=device)
    if i == 5:
        prefix, chunk = max(int(131_072 * scale), 1), max(int(8192 * scale), 1)
        return build_workload("prefill-131k+8k" + sfx, full, [prefix + chunk], [chunk], seed=4,
                              device=device, slack_blocks=64)
    raise ValueError(f"unknown config {i}")


# ----------------------------------------------------------------------------- token shards
def shard_visible(p: int, r: int, n_shards: int) -> int:
    """Local positions of shard r (global positions r, r + N, ...) visible from global position p."""
    return 0 if p < r else (p - r) // n_shards + 1


def shard_pools(wl: Workload, layout, pool: torch.Tensor, n_shards: int, *, seed: int, layer: int = 0):
    """Split a decode workload's context into N round-robin token shards, each in its own pool.

    Global position j of sequence b goes to shard r = j % N at local position
    j // N, in a fresh pool with its own (randomly permuted) block table; the
    record, indexer key and indexer scale bytes of each position are copied from
    ``pool`` (which must already hold every position, this step's included).
    One query token per sequence (at position seq_len - 1) is assumed.
    Returns, per shard, dict(layout, pool, block_table, seq_lens, max_ctx).
    """
    from . import layout_init  # the package's C-ABI binding

    d = wl.dims
    bs = d.block_size
    dev = pool.device
    rng = np.random.default_rng(seed)
    bt = wl.block_table.cpu().numpy()
    lens = wl.seq_lens.cpu().numpy()
    shards = []
    for r in range(n_shards):
        lr = [shard_visible(int(n) - 1, r, n_shards) for n in lens]
        nblk = [(x + bs - 1) // bs for x in lr]
        total = sum(nblk) + 1
        lay_r = layout_init(bs, d.n_layers, d.d_latent, d.d_rope, d.quant_tile, d.d_index, total, d.key_format)
        pool_r = torch.zeros(lay_r.pool_bytes, dtype=torch.uint8, device=dev)
        perm = rng.permutation(total)
        bt_r = np.zeros((len(lens), max(1, max(nblk))), dtype=np.int32)
        nxt = 0
        src, dst = [], []
        for b in range(len(lens)):
            bt_r[b, :nblk[b]] = perm[nxt:nxt + nblk[b]]
            nxt += nblk[b]
            i = np.arange(lr[b], dtype=np.int64)
            j = i * n_shards + r
            src.append(bt[b, j // bs].astype(np.int64) * bs + j % bs)
            dst.append(bt_r[b, i // bs].astype(np.int64) * bs + i % bs)
        src_all = torch.as_tensor(np.concatenate(src), device=dev)
        dst_all = torch.as_tensor(np.concatenate(dst), device=dev)
        for c0 in range(0, src_all.numel(), 1 << 16):   # bounded index tensors
            src, dst = src_all[c0:c0 + (1 << 16)], dst_all[c0:c0 + (1 << 16)]
            for name, unit in (("rec_off", layout.rec_stride), ("idx_key_off", layout.key_bytes), ("idx_scale_off", 4)):
                ar = torch.arange(unit, device=dev, dtype=torch.int64)
                s0 = (src // bs) * layout.block_stride + layer * layout.layer_stride + getattr(layout, name) + \
                    (src % bs) * unit
                d0 = (dst // bs) * lay_r.block_stride + layer * lay_r.layer_stride + getattr(lay_r, name) + \
                    (dst % bs) * unit
                pool_r[(d0[:, None] + ar).reshape(-1)] = pool[(s0[:, None] + ar).reshape(-1)]
        shards.append(dict(layout=lay_r, pool=pool_r, block_table=torch.as_tensor(bt_r, device=dev),
                           seq_lens=torch.as_tensor(np.asarray(lr, dtype=np.int32), device=dev),
                           max_ctx=max(1, max(lr))))
    return shards


# ----------------------------------------------------------------------------- host tier
def evict_records(layout, pool: torch.Tensor, blocks, *, chunk: int = 256):
    """Move the latent records of `blocks` (every layer) to pinned host memory.

    Returns (host_records uint8 pinned [n * n_layers * block_size * rec_stride],
    host_block_map int32 [num_blocks] on the pool's device: -1 = in the pool,
    h = host block h).  The moved regions are zeroed in the pool; indexer keys
    and scales stay.
    """
    dev = pool.device
    blocks = torch.as_tensor(np.asarray(blocks, dtype=np.int64), device=dev)
    per = layout.block_size * layout.rec_stride
    n = blocks.numel()
    host = torch.empty(n * layout.n_layers * per, dtype=torch.uint8).pin_memory()
    hmap = torch.full((layout.num_blocks,), -1, dtype=torch.int32, device=dev)
    hmap[blocks] = torch.arange(n, dtype=torch.int32, device=dev)
    ar = torch.arange(per, device=dev, dtype=torch.int64)
    view = host.view(n, layout.n_layers, per)  # host layout [block][layer][records]
    for c0 in range(0, n, chunk):
        b = blocks[c0:c0 + chunk]
        for layer in range(layout.n_layers):
            idx = ((b * layout.block_stride + layer * layout.layer_stride + layout.rec_off)[:, None] + ar).reshape(-1)
            view[c0:c0 + b.numel(), layer].copy_(pool[idx].reshape(b.numel(), per).cpu())
            pool[idx] = 0
    return host, hmap
