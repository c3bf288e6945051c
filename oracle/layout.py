"""Packed block-pool layout.

[AgentX "Hybrid KV cache management"]: every attention type shares one block
pool whose allocation unit is the page (block); the packed KV layout stores
all cache groups and layers of a block in one contiguous allocation instead of
one tensor per group.

reading: a block of ``block_size`` tokens holds, for each layer l in order,

    [bs latent records, stride rec_stride][bs indexer keys, key_bytes B][bs fp32 indexer scales]

each region starting on a 256-byte boundary of the block; the layer slice is
rounded up to 256 bytes and the block stride is n_layers times that.  A latent
record is

    [d_latent e4m3 codes][d_latent/quant_tile fp32 scales][d_rope bf16][pad to 16 B]

(656 bytes for d_latent=512, quant_tile=128, d_rope=64; 100 -> 112 bytes for
d_latent=64, quant_tile=64, d_rope=16).

reading (FP4 indexer keys, [AgentX "Hybrid KV cache management"]): with
``key_format="e2m1"`` an indexer key is d_index FP4 E2M1 codes packed two per
byte (key_bytes = d_index / 2 instead of d_index), so the key region and with
it the block shrink: 656 + 64 + 4 bytes per token instead of 656 + 128 + 4 for
the DeepSeek shape.
"""

from dataclasses import dataclass


def _round_up(x: int, m: int) -> int:
    return (x + m - 1) // m * m


@dataclass(frozen=True)
class PoolLayout:
    block_size: int
    n_layers: int
    d_latent: int
    d_rope: int
    quant_tile: int
    d_index: int
    num_blocks: int
    key_format: str = "e4m3"   # "e4m3": one byte per key element; "e2m1": two elements per byte

    def __post_init__(self):
        if self.key_format not in ("e4m3", "e2m1"):
            raise ValueError(f"unknown indexer key format {self.key_format!r}")
        if self.key_format == "e2m1" and self.d_index % 2:
            raise ValueError("packed E2M1 keys need an even d_index")

    @property
    def key_bytes(self) -> int:
        return self.d_index if self.key_format == "e4m3" else self.d_index // 2

    @property
    def n_scales(self) -> int:
        return self.d_latent // self.quant_tile

    @property
    def rec_bytes(self) -> int:
        return self.d_latent + 4 * self.n_scales + 2 * self.d_rope

    @property
    def rec_stride(self) -> int:
        return _round_up(self.rec_bytes, 16)

    @property
    def rec_off(self) -> int:
        return 0

    @property
    def idx_key_off(self) -> int:
        return _round_up(self.block_size * self.rec_stride, 256)

    @property
    def idx_scale_off(self) -> int:
        return _round_up(self.idx_key_off + self.block_size * self.key_bytes, 256)

    @property
    def layer_stride(self) -> int:
        return _round_up(self.idx_scale_off + 4 * self.block_size, 256)

    @property
    def block_stride(self) -> int:
        return self.n_layers * self.layer_stride

    @property
    def pool_bytes(self) -> int:
        return self.num_blocks * self.block_stride

    def record_offset(self, slot: int, layer: int) -> int:
        blk, off = divmod(int(slot), self.block_size)
        return blk * self.block_stride + layer * self.layer_stride + self.rec_off + off * self.rec_stride

    def index_key_offset(self, slot: int, layer: int) -> int:
        blk, off = divmod(int(slot), self.block_size)
        return blk * self.block_stride + layer * self.layer_stride + self.idx_key_off + off * self.key_bytes

    def index_scale_offset(self, slot: int, layer: int) -> int:
        blk, off = divmod(int(slot), self.block_size)
        return blk * self.block_stride + layer * self.layer_stride + self.idx_scale_off + off * 4
