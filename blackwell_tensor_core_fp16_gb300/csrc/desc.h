// Encoders shared by the host (unit tests, launch set-up) and the device (the kernels):
// the tcgen05 instruction descriptor, the shared-memory matrix descriptor, the 128-byte
// swizzle, the mbarrier ring's stage/phase sequence and the persistent tile order.
#pragma once

#include <cstdint>

#if defined(__CUDACC__)
#define GF16_HD __host__ __device__ __forceinline__ constexpr
#else
#define GF16_HD inline constexpr
#endif

namespace gf16 {

// ---------------------------------------------------------------------------------------------
// Instruction descriptor of tcgen05.mma .kind::f16 (dense), a 32-bit word:
//   bits  5:4   accumulator format       (1 = f32)
//   bits  9:7   A format                 (0 = f16, 1 = bf16)
//   bits 12:10  B format                 (0 = f16, 1 = bf16)
//   bit  15/16  A / B major              (0 = K-major)
//   bits 22:17  N >> 3
//   bits 28:24  M >> 4
// Everything else (sparsity, saturation, negation, shift) is zero.  For f16 x f16 -> f32 with
// M = N = 128 and both operands K-major this gives 0x08200010, the constant the page
// "TIRx Compiler Foundation" (section "Example: A GEMM Kernel") uses for its 128x128 tile.
// ---------------------------------------------------------------------------------------------
GF16_HD uint32_t make_idesc_f16(uint32_t M, uint32_t N, uint32_t ab_bf16)
{
    return (1u << 4) | ((ab_bf16 & 7u) << 7) | ((ab_bf16 & 7u) << 10) | (((N >> 3) & 0x3Fu) << 17) |
           (((M >> 4) & 0x1Fu) << 24);
}

// ---------------------------------------------------------------------------------------------
// Instruction descriptor of tcgen05.mma .kind::mxf8f6f4 with block scaling (E8M0 scales, one per
// 32 K elements), a 32-bit word:
//   bits  5:4   B scale-factor ID: the byte of each 32-bit scale column this MMA reads
//   bits  9:7   A format                 (0 = E4M3, 1 = E5M2)
//   bits 12:10  B format
//   bit  15/16  A / B major              (0 = K-major)
//   bits 22:17  N >> 3
//   bit  23     scale format             (1 = E8M0)
//   bits 28:24  M >> 4
//   bits 30:29  A scale-factor ID
// The IDs are left 0 here; the MMA issuer ORs in the K block (0-3) of each MMA.
// ---------------------------------------------------------------------------------------------
GF16_HD uint32_t make_idesc_mx(uint32_t M, uint32_t N, uint32_t fmt_a, uint32_t fmt_b)
{
    return ((fmt_a & 7u) << 7) | ((fmt_b & 7u) << 10) | (((N >> 3) & 0x3Fu) << 17) | (1u << 23) |
           (((M >> 4) & 0x1Fu) << 24);
}

GF16_HD uint32_t idesc_mx_with_sf_id(uint32_t idesc, uint32_t k_block)
{
    return idesc | ((k_block & 3u) << 4) | ((k_block & 3u) << 29);
}

// ---------------------------------------------------------------------------------------------
// The tiled layout of block scales (one E8M0 byte per row and per 32-element K block) that the
// kernels read.  Rows are grouped by 128 and K blocks by 4; each (row group, K-block group)
// pair is one contiguous 512-byte chunk, chunks ordered row-group-major.  Inside a chunk,
// row r = 32 q + l (l < 32, q < 4) and K block b (b < 4) sit at byte 16 l + 4 q + b: the 16
// bytes at 16 l are the 128-bit row l of a 32 x 128-bit block that tcgen05.cp .32x128b.warpx4
// copies into lane l of every 32-lane window of tensor memory, so tensor-memory column q holds
// rows 32 q .. 32 q + 31 and its byte b holds K block b.
// ---------------------------------------------------------------------------------------------
GF16_HD uint32_t mx_k_groups(uint32_t k_blocks) { return (k_blocks + 3u) / 4u; }

GF16_HD uint64_t mx_sf_offset(uint64_t row, uint32_t k_block, uint32_t k_groups)
{
    return ((row / 128u) * k_groups + k_block / 4u) * 512u + (row % 32u) * 16u +
           ((row % 128u) / 32u) * 4u + (k_block % 4u);
}

// Shared-memory descriptor of one 512-byte scale chunk as the source of tcgen05.cp .32x128b:
// 32 rows of 16 bytes, no swizzle, 8-row core matrices 128 bytes apart (both offset fields
// carry that stride; the copy is one core matrix wide).
GF16_HD uint64_t make_sf_desc(uint32_t smem_addr)
{
    uint64_t d = 0;
    d |= static_cast<uint64_t>((smem_addr & 0x3FFFFu) >> 4);
    d |= static_cast<uint64_t>(128u >> 4) << 16;
    d |= static_cast<uint64_t>(128u >> 4) << 32;
    d |= static_cast<uint64_t>(1u) << 46;
    return d;
}

// ---------------------------------------------------------------------------------------------
// Shared-memory matrix descriptor (64-bit) for a K-major operand tile stored with the 128-byte
// swizzle: rows of 64 fp16 (128 bytes), grouped in atoms of 8 rows = 1024 bytes.
//   bits 13:0   start address >> 4
//   bits 29:16  leading-dimension byte offset >> 4 (not used by swizzled K-major tiles; 1)
//   bits 45:32  stride-dimension byte offset >> 4  (distance between 8-row atoms: 1024 B)
//   bits 48:46  fixed 0b001 (the tcgen05 descriptor version)
//   bits 51:49  base offset (0: every tile starts on a 1024-byte boundary)
//   bit  52     leading-dimension mode (0: relative)
//   bits 63:61  swizzle mode (2 = 128-byte swizzle)
// Stepping along K inside the 128-byte row (16 fp16 = 32 bytes per MMA) adds 32 bytes to the
// start address, i.e. 2 to the low field: the swizzle is a function of the final address bits,
// so the same XOR pattern the TMA wrote is applied to the shifted address.
// ---------------------------------------------------------------------------------------------
GF16_HD uint64_t make_smem_desc_sw128(uint32_t smem_addr, uint32_t sbo_bytes)
{
    uint64_t d = 0;
    d |= static_cast<uint64_t>((smem_addr & 0x3FFFFu) >> 4);
    d |= static_cast<uint64_t>(1u) << 16;
    d |= static_cast<uint64_t>((sbo_bytes >> 4) & 0x3FFFu) << 32;
    d |= static_cast<uint64_t>(1u) << 46;
    d |= static_cast<uint64_t>(2u) << 61;
    return d;
}

// ---------------------------------------------------------------------------------------------
// 128-byte swizzle of a byte offset inside a 1024-byte-aligned tile whose rows are 128 bytes:
// the 16-byte chunk index (bits 6:4) is XORed with the row index modulo 8 (bits 9:7).  For an
// (8, 64) fp16 tile this is the element map addr = 64*i + 8*(q xor i) + r with q = j / 8 and
// r = j mod 8, the worked example of the page "chapter_tirx_layout_api" (section "示例：对
// (8, 64) float16 Tile 应用 128B Swizzle"), there derived from per_element = 3,
// swizzle_len = 3, atom_len = 3.
// ---------------------------------------------------------------------------------------------
GF16_HD uint32_t sw128(uint32_t byte_offset)
{
    return byte_offset ^ ((byte_offset >> 3) & 0x70u);
}

// ---------------------------------------------------------------------------------------------
// The mbarrier ring.  Iteration `it` (counted across all tiles a CTA processes, never reset)
// uses stage it % S and waits for the phase of parity (it / S) & 1 on that stage's "full"
// barrier; the producer waits on the stage's "empty" barrier with the opposite parity, so its
// first pass over the ring proceeds at once.  Carrying `it` across tiles removes the
// requirement that a tile's K-iteration count be a multiple of 2*S.
// ---------------------------------------------------------------------------------------------
struct RingPos {
    uint32_t stage;
    uint32_t parity;
};

GF16_HD RingPos ring_pos(uint32_t it, uint32_t stages)
{
    return RingPos{it % stages, (it / stages) & 1u};
}

// ---------------------------------------------------------------------------------------------
// Persistent tile order with grouped rasterisation: tiles are numbered so that consecutive
// numbers walk down a group of `group` tile-rows inside one tile-column, then move to the next
// column; groups follow each other down the M dimension.  A wave of CTAs therefore shares a
// few B column bands and a few A row bands, which keeps both in L2 (the l2_group_size idea of
// the page "TIRx 与高性能GEMM (上)", section "Step 6").
// ---------------------------------------------------------------------------------------------
struct TileCoord {
    uint32_t m_blk;
    uint32_t n_blk;
};

GF16_HD TileCoord tile_coord(uint32_t t, uint32_t num_m, uint32_t num_n, uint32_t group)
{
    const uint32_t per_group = group * num_n;
    const uint32_t g = t / per_group;
    const uint32_t first_m = g * group;
    const uint32_t left = num_m - first_m;
    const uint32_t gsize = left < group ? left : group;
    const uint32_t r = t - g * per_group;
    return TileCoord{first_m + r % gsize, r / gsize};
}

// ---------------------------------------------------------------------------------------------
// Work split of the persistent kernel with a stream-K tail.  T tiles, U persistent units (CTAs
// or CTA pairs), KB k-blocks per tile, and R tail tiles (R = 0: pure data-parallel).
//   * data-parallel part: tiles [0, T - R); unit c takes c, c + U, ... (T - R is a multiple of U
//     when R > 0, so every unit gets W = (T - R) / U of them);
//   * stream-K part: the R tail tiles' k-blocks, numbered x = r * KB + kb over [0, R * KB), are
//     cut into S contiguous ranges [lo_c, hi_c) with lo_c = floor(c * R * KB / S), one for each
//     of units 0 .. S-1 (S <= U); each range is split at tile boundaries into pieces.  With
//     R <= S a range is at most KB long, so a unit has at most two pieces, and a tail tile has
//     at most ceil(S / R) + 1 contributors.
// A piece that does not cover its whole tile is "partial": its fp32 accumulator is summed with
// the other pieces of the tile by the piece that starts the tile.
//
// Half-width tail (H > 0, then R = 0): the last H tiles (the partial wave, or every tile when
// there are fewer tiles than units), each cut into two items of half its columns, so that the
// 2 H <= U items run in about half a tile's time: unit c < 2 H takes half c % 2 of tail tile
// T - H + c / 2 after its data-parallel tiles [0, T - H), a multiple of U.
// ---------------------------------------------------------------------------------------------
struct WorkSplit {
    uint32_t T, U, KB, R;
    uint32_t S;      // units sharing the stream-K k-blocks (units S .. U-1 get none); S <= U
    uint32_t H = 0;  // tail tiles cut into two half-width items (0: none)
};

struct WorkItem {
    uint32_t tile;      // tile number in the grouped order
    uint32_t kb0;       // first k-block
    uint32_t kb1;       // one past the last k-block
    uint32_t piece;     // 0 or 1 for stream-K pieces (workspace slot), unused otherwise
    uint32_t partial;   // 1 if the piece's accumulator must be combined with others
    uint32_t half = 0;  // 0: the whole tile; 1, 2: its first or second half of the columns
};

GF16_HD uint32_t sk_lo(const WorkSplit& w, uint32_t c)
{
    const uint32_t cc = c < w.S ? c : w.S;
    return static_cast<uint32_t>((static_cast<uint64_t>(cc) * w.R * w.KB) / w.S);
}

GF16_HD uint32_t dp_tiles_of(const WorkSplit& w, uint32_t c)
{
    const uint32_t dp = w.T - w.R - w.H;
    if (w.R > 0 || w.H > 0) return dp / w.U;
    return c < dp ? (dp - c + w.U - 1) / w.U : 0u;
}

GF16_HD uint32_t half_items_of(const WorkSplit& w, uint32_t c)
{
    return c < 2u * w.H ? 1u : 0u;
}

GF16_HD uint32_t sk_pieces_of(const WorkSplit& w, uint32_t c)
{
    if (w.R == 0) return 0u;
    const uint32_t lo = sk_lo(w, c), hi = sk_lo(w, c + 1);
    return hi > lo ? (hi - 1) / w.KB - lo / w.KB + 1 : 0u;
}

GF16_HD uint32_t items_of(const WorkSplit& w, uint32_t c)
{
    return dp_tiles_of(w, c) + sk_pieces_of(w, c) + half_items_of(w, c);
}

// Total k-block iterations of unit c (the pipeline counters run over these).
GF16_HD uint32_t iterations_of(const WorkSplit& w, uint32_t c)
{
    return dp_tiles_of(w, c) * w.KB + (w.R ? sk_lo(w, c + 1) - sk_lo(w, c) : 0u) +
           half_items_of(w, c) * w.KB;
}

GF16_HD WorkItem work_item(const WorkSplit& w, uint32_t c, uint32_t idx)
{
    const uint32_t ndp = dp_tiles_of(w, c);
    if (idx < ndp) return WorkItem{c + idx * w.U, 0u, w.KB, 0u, 0u};
    if (w.H > 0) return WorkItem{w.T - w.H + c / 2u, 0u, w.KB, 0u, 0u, 1u + c % 2u};
    const uint32_t j = idx - ndp;
    const uint32_t lo = sk_lo(w, c), hi = sk_lo(w, c + 1);
    const uint32_t r = lo / w.KB + j;
    const uint32_t start = (j == 0 ? lo : r * w.KB) - r * w.KB;
    const uint32_t end = (hi < (r + 1) * w.KB ? hi : (r + 1) * w.KB) - r * w.KB;
    const uint32_t partial = (start != 0u || end != w.KB) ? 1u : 0u;
    return WorkItem{w.T - w.R + r, start, end, j, partial};
}

// The unit whose stream-K range holds tail k-block x.
GF16_HD uint32_t sk_unit_of(const WorkSplit& w, uint32_t x)
{
    return static_cast<uint32_t>(((static_cast<uint64_t>(x) + 1u) * w.S - 1u) /
                                 (static_cast<uint64_t>(w.R) * w.KB));
}

}  // namespace gf16
