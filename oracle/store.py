"""FP8 KV store into the packed pool, and record readers.

[GLM-5.3 "Config and numbers", "How to try"]: the KV cache is FP8 (1M tokens
take 53.4 GiB).  [AgentX "Hybrid KV cache management"]: one packed allocation
per block holds every cache group.

reading (quantisation): for each token, the bf16 latent vector is cut into
tiles of ``quant_tile`` elements.  Per tile:
    amax  = max |x|                          (exact)
    scale = fp32(amax / 448)                 (one IEEE fp32 division, RNE)
    scale = 1.0 if scale == 0
    code  = e4m3_rne_satfinite(fp32(x / scale))
The rope part (bf16) and the caller-supplied indexer key (e4m3 bytes, or
packed e2m1 bytes for a layout with FP4 keys) and indexer scale (fp32) are
copied verbatim.  ``slot_mapping[t] == -1`` skips
token t.  Dequantisation of a code is fp32(decode(code) * scale).

fp32 division and multiplication are evaluated in float64 and rounded once to
float32: for p = 24-bit operands a q >= 2p+2 = 50-bit intermediate gives the
correctly rounded p-bit result (no double-rounding error), and float64 has 53.
"""

import numpy as np

from .fp4 import e2m1_decode, e2m1_unpack
from .fp8 import e4m3_decode, e4m3_encode, E4M3_MAX
from .layout import PoolLayout


def bf16_bits_to_f64(bits) -> np.ndarray:
    """bf16 bit patterns (uint16) -> exact float64 values."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16
    return b.view(np.float32).astype(np.float64)


def quantize_latent(latent_bits, quant_tile: int):
    """bf16 latent [T, D_L] -> (codes uint8 [T, D_L], scales fp32 [T, D_L/quant_tile])."""
    x = bf16_bits_to_f64(latent_bits)
    t, d = x.shape
    tiles = x.reshape(t, d // quant_tile, quant_tile)
    amax = np.abs(tiles).max(axis=2)
    scale = (amax / E4M3_MAX).astype(np.float32)
    scale = np.where(scale == 0, np.float32(1.0), scale).astype(np.float32)
    q = (tiles / scale.astype(np.float64)[:, :, None]).astype(np.float32)
    codes = e4m3_encode(q).reshape(t, d)
    return codes, scale


def _offsets(layout: PoolLayout, slots, layer: int, region: str) -> np.ndarray:
    slots = np.asarray(slots, dtype=np.int64)
    blk, off = slots // layout.block_size, slots % layout.block_size
    base = blk * layout.block_stride + layer * layout.layer_stride
    if region == "record":
        return base + layout.rec_off + off * layout.rec_stride
    if region == "key":
        return base + layout.idx_key_off + off * layout.key_bytes
    return base + layout.idx_scale_off + off * 4


def kvpack_store(layout: PoolLayout, pool: np.ndarray, layer: int, latent_bits, rope_bits,
                 idx_k, idx_scale, slot_mapping) -> None:
    """Write new tokens' records into ``pool`` (uint8, modified in place)."""
    slots = np.asarray(slot_mapping, dtype=np.int64)
    keep = slots >= 0
    codes, scales = quantize_latent(np.asarray(latent_bits)[keep], layout.quant_tile)
    rope = np.ascontiguousarray(np.asarray(rope_bits, dtype=np.uint16)[keep])
    idx_k = np.asarray(idx_k, dtype=np.uint8)[keep]
    idx_scale = np.ascontiguousarray(np.asarray(idx_scale, dtype=np.float32)[keep])
    slots = slots[keep]
    d_l, n_s, d_r, d_i = layout.d_latent, layout.n_scales, layout.d_rope, layout.key_bytes
    rec = _offsets(layout, slots, layer, "record")[:, None]
    pool[rec + np.arange(d_l)] = codes
    pool[rec + d_l + np.arange(4 * n_s)] = np.ascontiguousarray(scales).view(np.uint8).reshape(-1, 4 * n_s)
    pool[rec + d_l + 4 * n_s + np.arange(2 * d_r)] = rope.view(np.uint8).reshape(-1, 2 * d_r)
    key = _offsets(layout, slots, layer, "key")[:, None]
    pool[key + np.arange(d_i)] = idx_k
    sc = _offsets(layout, slots, layer, "scale")[:, None]
    pool[sc + np.arange(4)] = idx_scale.view(np.uint8).reshape(-1, 4)


def read_record(layout: PoolLayout, pool: np.ndarray, layer: int, slots):
    """Dequantised latent [n, D_L] (fp32 values held in float64) and rope [n, D_R] (float64)."""
    d_l, n_s, d_r = layout.d_latent, layout.n_scales, layout.d_rope
    rec = _offsets(layout, slots, layer, "record")[:, None]
    codes = pool[rec + np.arange(d_l)]
    scales = np.ascontiguousarray(pool[rec + d_l + np.arange(4 * n_s)]).view(np.float32)
    vals = e4m3_decode(codes).reshape(-1, n_s, layout.quant_tile) * scales.astype(np.float64)[:, :, None]
    lat = vals.reshape(-1, d_l).astype(np.float32).astype(np.float64)   # fp32(decode(code) * scale)
    rope_bits = np.ascontiguousarray(pool[rec + d_l + 4 * n_s + np.arange(2 * d_r)]).view(np.uint16)
    return lat, bf16_bits_to_f64(rope_bits)


def read_index_key(layout: PoolLayout, pool: np.ndarray, layer: int, slots):
    """Indexer keys (decoded e4m3 or e2m1, float64) [n, D_I] and their fp32 scales [n] (float64)."""
    key = _offsets(layout, slots, layer, "key")[:, None]
    raw = pool[key + np.arange(layout.key_bytes)]
    keys = e4m3_decode(raw) if layout.key_format == "e4m3" else e2m1_decode(e2m1_unpack(raw))
    sc = _offsets(layout, slots, layer, "scale")[:, None]
    scales = np.ascontiguousarray(pool[sc + np.arange(4)]).view(np.float32)[:, 0]
    return keys, scales.astype(np.float64)
