/*
 * gemm_f16.h -- C ABI of the GB300 (sm_103a) fp16 GEMM library libgemm_f16.so.
 *
 * The operation (page "TIRx 与高性能GEMM (上)", section "从 GEMM 公式到数据路径"):
 *
 *     D = A * B^T,   D[i][j] = sum_{k < K} A[i][k] * B[j][k]
 *
 * A is M x K, B is N x K (the weight layout: each row of B is one output feature, K
 * contiguous, so the transpose is a property of the storage and no data is moved), D is M x N.
 * All three are IEEE binary16, row-major and dense (leading dimensions K, K and N).  Products
 * are accumulated in fp32 in Tensor Memory; each output is rounded to fp16 with
 * round-to-nearest-even (page "TIRx Compiler Foundation", section "Example: A GEMM Kernel":
 * the accumulator is converted to FP16 with cvt.rn before the store).
 *
 * Memory: the caller owns A, B and D (and the optional workspace of gemm_f16_nt_ws), which must
 * be device memory of the current CUDA device.  The library allocates no device memory, keeps no
 * pointer beyond a call, and only caches host-side objects (TMA descriptors, device
 * properties).  D is overwritten, never read.
 *
 * Asynchrony: every compute entry point enqueues work on `stream` and returns; it does not
 * synchronise.  Errors that need the GPU to detect (a bounded wait that ran out) are reported
 * by gemm_f16_check_status().
 *
 * Stream order: the persistent kernels (every variant but GEMM_F16_VARIANT_TILE) are launched
 * with programmatic stream serialization.  A launch may start its set-up on SMs that the kernel
 * before it on the stream has already left, but it reads and writes no global memory until that
 * kernel has completed and its writes are visible, so results are ordered exactly as on a plain
 * stream.  Setting the environment variable GEMM_F16_PDL=0 (read once per process) launches them
 * the plain way.
 *
 * Thread safety: entry points may be called from several host threads at once.
 */
#ifndef GEMM_F16_H
#define GEMM_F16_H

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Status codes returned by every entry point that can fail. */
#define GEMM_F16_OK 0
/* A null pointer with a non-empty operand, a negative size, or a size above 2^31 - 1. */
#define GEMM_F16_ERR_INVALID_ARG 1
/* A shape or pointer the tensor-memory-access path cannot address: K or N not a multiple of 8
 * (row strides must be multiples of 16 bytes), or A, B or D not 16-byte aligned.  There is no
 * fallback path; the call does nothing. */
#define GEMM_F16_ERR_UNSUPPORTED 2
/* A CUDA runtime or driver call failed; gemm_f16_last_error() describes it. */
#define GEMM_F16_ERR_CUDA 3
/* A kernel gave up a bounded wait (its pipeline did not make progress within the limit);
 * D is unspecified.  Returned by gemm_f16_check_status() only. */
#define GEMM_F16_ERR_TIMEOUT 4

/* Kernel variants (gemm_f16_nt_variant).  All compute the same D. */
#define GEMM_F16_VARIANT_AUTO 0       /* choose by shape and device */
#define GEMM_F16_VARIANT_TILE 1       /* one 128 x n tile per CTA, two-stage K loop; n is the
                                         narrowest of 16, 32, 64 whose grid fits one wave, else
                                         128 (fp16 only; chosen for short K and at most one wave
                                         of 128 x 128 tiles) */
#define GEMM_F16_VARIANT_WS_128x256 2 /* persistent, warp-specialised, 1 CTA per 128x256 tile */
#define GEMM_F16_VARIANT_WS_PAIR 3    /* persistent, warp-specialised, CTA pair per 256x256 */
#define GEMM_F16_VARIANT_WS_128x128 4 /* persistent, warp-specialised, 1 CTA per 128x128 tile */
#define GEMM_F16_VARIANT_WS_PAIR_DIRECT 5 /* as WS_PAIR, 7 stages, epilogue stores from registers */
#define GEMM_F16_VARIANT_WS_PAIR_256x192 6 /* as WS_PAIR with 256x192 tiles; explicit only: 0.91-0.99
                                             of WS_PAIR on every shape measured */
#define GEMM_F16_NUM_VARIANTS 7

/*
 * D = A * B^T for fp16 A (M x K), B (N x K), D (M x N), fp32 accumulation, on `stream`.
 *
 * A, B, D: device pointers (binary16 elements), 16-byte aligned.
 * M, N, K: sizes, 0 <= each <= 2^31 - 1; K % 8 == 0 and N % 8 == 0.
 * stream:  the CUDA stream to enqueue on (0 is the legacy default stream).
 *
 * M == 0 or N == 0: nothing to compute; returns GEMM_F16_OK without touching any pointer.
 * K == 0: D is the empty sum, all zeros (filled with cudaMemsetAsync).
 * Returns a GEMM_F16_* status; on any status other than GEMM_F16_OK nothing was enqueued.
 */
int gemm_f16_nt(const void* A, const void* B, void* D, int64_t M, int64_t N, int64_t K,
                cudaStream_t stream);

/* Same operation with an explicit kernel variant (GEMM_F16_VARIANT_*), for benchmarking and
 * cross-checking; GEMM_F16_VARIANT_AUTO is what gemm_f16_nt uses.  An unknown variant is
 * GEMM_F16_ERR_INVALID_ARG. */
int gemm_f16_nt_variant(const void* A, const void* B, void* D, int64_t M, int64_t N, int64_t K,
                        cudaStream_t stream, int variant);

/* Element types and activations of gemm_f16_nt_fused. */
#define GEMM_F16_DTYPE_F16 0  /* IEEE binary16 */
#define GEMM_F16_DTYPE_BF16 1 /* bfloat16 */
#define GEMM_F16_ACT_NONE 0
#define GEMM_F16_ACT_RELU 1   /* max(y, 0) */
#define GEMM_F16_ACT_GELU 2   /* y * Phi(y) = y/2 * (1 + erf(y / sqrt 2)), the exact form */

/*
 * A linear layer: D = act(A * B^T + bias), for fp16 or bf16 data.  bf16 inputs use the same
 * tensor-core path as fp16 (tcgen05.mma .kind::f16 with the instruction descriptor's A/B format
 * set to bf16); the page "TIRx" (section "SM90a 支持具体补了什么") names FP16 and BF16 inputs with
 * FP32 accumulation, and the page "TIRx 与高性能GEMM (上)" motivates the GEMM by linear layers.
 *
 * dtype:      GEMM_F16_DTYPE_F16 or GEMM_F16_DTYPE_BF16, for A, B, D and bias alike.
 * bias:       N elements (one per output column), 16-byte aligned, or null for none.
 * activation: GEMM_F16_ACT_*.
 * variant:    GEMM_F16_VARIANT_AUTO or one of the persistent variants (2, 3, 4).
 * workspace:  as gemm_f16_nt_ws (may be null).
 * The bias and the activation are applied in fp32 to the fp32 sum; the result is then rounded
 * once (round to nearest even) to the output type.  GELU is evaluated with a published
 * Chebyshev fit of erfc (Numerical Recipes, section 6.2), within 2e-7 plus one fp32 rounding
 * of the exact GELU for |y| <= 10 before that rounding.  K must be at least 1.  Other rules and return codes as
 * gemm_f16_nt.
 */
int gemm_f16_nt_fused(const void* A, const void* B, void* D, int64_t M, int64_t N, int64_t K,
                      int dtype, const void* bias, int activation, int variant, void* workspace,
                      size_t workspace_bytes, cudaStream_t stream);

/*
 * D = A * B^T with a caller-provided workspace, which lets the persistent kernels run the tiles
 * of the last, partial wave "stream-K" once gemm_f16_set_stream_k(1) has turned that on: the
 * tail tiles' k-blocks are split evenly over the CTAs; the CTA whose piece starts a tile
 * finishes it, adding the other pieces' fp32 partial sums (which their CTAs park in the
 * workspace, raising a flag each) in k order to its own, so the result does not depend on
 * timing.  With stream-K off (the default) the workspace is not used.
 *
 * workspace:       device memory, 256-byte aligned, at least gemm_f16_workspace_bytes(...) bytes
 *                  (or null / too small: the call runs without the stream-K tail).  The library
 *                  clears the workspace's 8 KiB header (flags and their bookkeeping) with
 *                  cudaMemsetAsync on `stream` before each stream-K launch and overwrites the
 *                  rest; nothing needs initialising.  Launches that share a workspace must not
 *                  overlap on the GPU (use one workspace per stream).
 * Everything else is as gemm_f16_nt.  The result differs from gemm_f16_nt's only in the order of
 * the fp32 additions of the tail tiles (both within the tolerance of an fp32 accumulation).
 */
int gemm_f16_nt_ws(const void* A, const void* B, void* D, int64_t M, int64_t N, int64_t K,
                   void* workspace, size_t workspace_bytes, cudaStream_t stream);

/* gemm_f16_nt_ws with an explicit variant (GEMM_F16_VARIANT_*). */
int gemm_f16_nt_ex(const void* A, const void* B, void* D, int64_t M, int64_t N, int64_t K,
                   int variant, void* workspace, size_t workspace_bytes, cudaStream_t stream);

/* Whether later launches of this process that have a workspace (gemm_f16_nt_ws, _ex, _fused,
 * gemm_f16_nt_noalloc) run the stream-K tail: 1 on, 0 off (the default).  Off by default because
 * on GB300 it measured slower than the data-parallel schedule on every workload tried (2048^3,
 * 3000x5000x1000, 8192^3, the MLP shape: 0.6-70% more time): parking a CTA's 128 KB of fp32
 * partial sums and reading them back costs more than the idle part of the last wave.  Returns
 * GEMM_F16_OK, or GEMM_F16_ERR_INVALID_ARG for any other value.  Host-only. */
int gemm_f16_set_stream_k(int enable);

/*
 * D = A * B^T without allocating anything, for callers that cannot allocate device memory:
 * servers that hand all device memory to their own pool at start-up and forbid any other
 * allocation, plug-ins running inside a host program that owns every allocation, and
 * latency-bound loops that cannot afford cudaMalloc's implicit synchronisation.  The GEMM pages
 * have no counterpart to this entry point; it is a deployment convenience.
 *
 * It computes what gemm_f16_nt_ws computes, with the stream-K workspace (when stream-K is on)
 * taken from a fixed 40 MiB array of device memory that the library reserves on every device
 * that loads it, for the life of the process.  The caller passes A, B and D as for gemm_f16_nt.
 * Nothing else is allocated: no cudaMalloc, cudaFree or allocating library routine is called.
 *
 * The first call on each device looks up the array's device address (cudaGetSymbolAddress) with
 * that device current; make that first call before any stream capture that uses this entry
 * point.  Every call shares the one array and finds the previous call's contents in it: the
 * array starts at zero and every launch leaves its 8 KiB header consistent (each launch clears
 * the flags the next one uses), so no clearing copy runs before a launch.  Calls that
 * overlap on the GPU (on different streams) race on the array and give wrong results: serialise
 * them.  A shape whose stream-K workspace would exceed the array (not possible on a 152-SM
 * GB300, whose largest request is about 38 MiB; possible on a GPU with many more SMs) runs the
 * plain data-parallel schedule instead, which needs no workspace: the result is the same, only
 * the last partial wave is not split.  Errors are those of gemm_f16_nt.
 */
int gemm_f16_nt_noalloc(const void* A, const void* B, void* D, int64_t M, int64_t N, int64_t K,
                        cudaStream_t stream);

/* Size in bytes of the fixed array gemm_f16_nt_noalloc uses (40 MiB).  Host-only. */
size_t gemm_f16_noalloc_scratch_bytes(void);

/* Workspace bytes gemm_f16_nt_ws / gemm_f16_nt_ex need for this shape and variant on the current
 * device (0: the shape gets no stream-K tail, or stream-K is off).  At most 8 KiB + units x
 * CTAs per unit x 128 x 256 x 4 bytes (about 19 MiB on a 152-SM GPU).  Queries the device;
 * launches nothing. */
int gemm_f16_workspace_bytes(int64_t M, int64_t N, int64_t K, int variant, size_t* bytes);

/* The variant GEMM_F16_VARIANT_AUTO picks for this shape on a device with `num_sms`
 * multiprocessors.  Host-only; needs no GPU. */
int gemm_f16_choose_variant(int64_t M, int64_t N, int64_t K, int num_sms);

/* Synchronise `stream`, then read and clear the device status word of the current device.
 * Returns GEMM_F16_OK, GEMM_F16_ERR_TIMEOUT (a kernel gave up a bounded wait; *bits, if not
 * null, receives which roles did) or GEMM_F16_ERR_CUDA. */
int gemm_f16_check_status(cudaStream_t stream, uint32_t* bits);

/* Wall-clock limit of each bounded wait inside the kernels, for launches made after the call
 * (default: GEMM_F16_WAIT_TIMEOUT_MS, else 4000 ms).  A wait that runs out makes the kernel stop
 * cleanly and report GEMM_F16_ERR_TIMEOUT through gemm_f16_check_status. */
int gemm_f16_set_wait_timeout_ms(uint32_t ms);

/* Testing hook for the failure path, process-wide, for launches made after the call.  mode 1:
 * the kernels' load producer issues no copies, so the first wait for operand data can only run
 * out (nothing asynchronous is left in flight; the kernel reports TIMEOUT and exits cleanly);
 * mode 0: normal operation.  Never set it outside tests. */
int gemm_f16_set_fault_injection(int mode);

/* Description of the last error on the calling thread ("" if none).  The string stays valid
 * until the thread's next call into the library. */
const char* gemm_f16_last_error(void);

/* Library version, major * 10000 + minor * 100 + patch. */
int gemm_f16_version(void);

/* ---- host-side encoders (no GPU needed; used by the unit tests) -------------------------- */

/* Static description of a variant's tiling.  Returns GEMM_F16_OK or GEMM_F16_ERR_INVALID_ARG. */
typedef struct gemm_f16_variant_info {
    int32_t cta_group;      /* CTAs per tile (1, or 2 for a CTA pair) */
    int32_t block_m;        /* output rows per tile */
    int32_t block_n;        /* output columns per tile */
    int32_t block_k;        /* K per pipeline stage */
    int32_t stages;         /* shared-memory pipeline stages */
    int32_t threads;        /* threads per CTA */
    int32_t smem_bytes;     /* dynamic shared memory per CTA */
    int32_t tmem_cols;      /* Tensor Memory columns per CTA */
    int32_t stage_tx_bytes; /* bytes a stage's "full" barrier expects (both CTAs of a pair) */
    int32_t persistent;     /* 1 if CTAs loop over tiles */
} gemm_f16_variant_info;

int gemm_f16_get_variant_info(int variant, gemm_f16_variant_info* out);

/* tcgen05.mma .kind::f16 instruction descriptor: fp32 accumulator, A and B both fp16
 * (ab_bf16 = 0) or both bf16 (1), K-major, M x N.  For M = N = 128, fp16: 0x08200010. */
uint32_t gemm_f16_idesc(uint32_t M, uint32_t N, uint32_t ab_bf16);

/* Shared-memory matrix descriptor of a K-major, 128-byte-swizzled operand tile at shared
 * address `smem_addr` whose 8-row atoms are `sbo_bytes` apart. */
uint64_t gemm_f16_smem_desc_sw128(uint32_t smem_addr, uint32_t sbo_bytes);

/* Byte offset after the 128-byte swizzle of byte offset `off` inside a 1024-byte-aligned tile
 * with 128-byte rows. */
uint32_t gemm_f16_sw128(uint32_t off);

/* Tile number t -> (m_blk, n_blk) in the persistent schedule's grouped order. */
void gemm_f16_tile_coord(uint32_t t, uint32_t num_m, uint32_t num_n, uint32_t group,
                         uint32_t* m_blk, uint32_t* n_blk);

/* Pipeline iteration `it` -> ring stage and the parity of the "full" phase it waits for. */
void gemm_f16_ring_pos(uint32_t it, uint32_t stages, uint32_t* stage, uint32_t* parity);

/* Raster group size (tile-rows walked together) the library launches with for tiles of `mma_m`
 * rows, depth K of `elem_bytes`-byte elements and an L2 of `l2_bytes`: the largest power of two up
 * to 16 whose G row bands of A (mma_m x K elements each) fit in a third of L2.  The environment
 * variable GEMM_F16_GROUP (1..64), read once per process, overrides it. */
uint32_t gemm_f16_raster_group(int64_t mma_m, int64_t K, int64_t elem_bytes, int64_t l2_bytes);

/* The persistent kernels' work split (host copies of the device arithmetic).  `tiles` output
 * tiles of `k_blocks` k-blocks each on `units` CTAs (or CTA pairs), of which the last `tail` run
 * stream-K (0: none).  gemm_f16_sk_tail_tiles: the tail the library chooses.
 * gemm_f16_sk_items: work items of one unit.  gemm_f16_sk_item: item `idx` of `unit` as
 * {tile, first k-block, end k-block, piece 0/1, partial 0/1}.  gemm_f16_sk_unit_of: the unit
 * whose stream-K range holds tail k-block x (x counts k-blocks over the tail tiles). */
int64_t gemm_f16_sk_tail_tiles(int64_t tiles, int64_t units, int64_t k_blocks);
uint32_t gemm_f16_sk_items(uint32_t tiles, uint32_t units, uint32_t k_blocks, uint32_t tail,
                           uint32_t unit);
void gemm_f16_sk_item(uint32_t tiles, uint32_t units, uint32_t k_blocks, uint32_t tail,
                      uint32_t unit, uint32_t idx, uint32_t out[5]);
uint32_t gemm_f16_sk_unit_of(uint32_t tiles, uint32_t units, uint32_t k_blocks, uint32_t tail,
                             uint32_t x);

/* The half-width tail (without stream-K): the tiles of the last, partial wave (all tiles when
 * there are fewer than `units`) each run as two items of half the tile's columns, when those fit
 * in one wave (2 x tail <= units).  gemm_f16_half_tail_tiles: that tail (0: none).
 * gemm_f16_half_items / gemm_f16_half_item: as gemm_f16_sk_items / _item for a split whose last
 * `half` tiles are cut this way; an item is {tile, first k-block, end k-block, half: 0 the whole
 * tile, 1 or 2 its first or second half of the columns}. */
int64_t gemm_f16_half_tail_tiles(int64_t tiles, int64_t units);
uint32_t gemm_f16_half_items(uint32_t tiles, uint32_t units, uint32_t k_blocks, uint32_t half,
                             uint32_t unit);
void gemm_f16_half_item(uint32_t tiles, uint32_t units, uint32_t k_blocks, uint32_t half,
                        uint32_t unit, uint32_t idx, uint32_t out[4]);

/* ---- block-scaled FP8 GEMM (MX formats) ------------------------------------------------------
 *
 * The operation (page "TIRx Layout API", sections "示例：Blackwell Tensor Memory" and
 * "Scale Factor 布局": a block-scaled FP8 GEMM whose MMA reads 8-bit scale factors kept in
 * tensor memory next to two accumulator stages, replicated into every 32-lane window).  The
 * pages fix neither the element formats nor the block length; this library implements the
 * OCP Microscaling reading that the tensor cores' mxf8f6f4 kind computes:
 *
 *     D[i][j] = sum_{k < K} (A[i][k] * 2^(SA[i][k/32] - 127)) * (B[j][k] * 2^(SB[j][k/32] - 127))
 *
 * A (M x K) and B (N x K) hold FP8 codes, row-major and dense (leading dimension K bytes), each
 * in E4M3 or E5M2 (chosen per operand).  SA and SB hold one E8M0 code (a biased exponent; 255
 * is NaN) per row and per block of 32 consecutive K elements, so K must be a multiple of 32.
 * The sums are accumulated in fp32 in tensor memory, then optionally act(sum + bias[j]) as in
 * gemm_f16_nt_fused, and rounded to fp16 or bf16 (round to nearest even) into D (M x N,
 * row-major, leading dimension N).
 *
 * Scale layout.  The kernels read SA and SB in a tiled layout, not row-major: rows in groups of
 * 128 and K blocks in groups of 4 form 512-byte chunks, ordered row-group-major; scale (r, b)
 * lives at byte
 *     ((r / 128) * ceil(K/128) + b / 4) * 512 + (r % 32) * 16 + ((r % 128) / 32) * 4 + b % 4
 * (gemm_mxf8_sf_offset computes it).  A buffer holds gemm_mxf8_scale_bytes(rows, K) bytes;
 * gemm_mxf8_pack_scales converts a row-major rows x K/32 array into it.  Padding bytes (rows
 * past the last full group, K blocks past K/32) are read: those of padded rows only reach
 * outputs that are never written, but those of padded K blocks multiply the zeros the K tail is
 * filled with, so they must not hold 255 (NaN); the pack routine writes 127 (1.0) there.
 *
 * Ownership, asynchrony and errors as for gemm_f16_nt; D is overwritten, never read.
 */
#define GEMM_MXF8_E4M3 0 /* 1 sign, 4 exponent (bias 7), 3 fraction bits; no infinities */
#define GEMM_MXF8_E5M2 1 /* 1 sign, 5 exponent (bias 15), 2 fraction bits; IEEE-like */

#define GEMM_MXF8_VARIANT_AUTO 0
#define GEMM_MXF8_VARIANT_128x128 1      /* persistent, warp-specialised, 1 CTA per 128x128 tile */
#define GEMM_MXF8_VARIANT_PAIR_256x128 2 /* persistent, warp-specialised, CTA pair per 256x128 */
#define GEMM_MXF8_VARIANT_PAIR_256x192 3 /* persistent, warp-specialised, CTA pair per 256x192 */
#define GEMM_MXF8_VARIANT_PAIR_256x256 4 /* as the pair, 256x256 tiles, one TMEM accumulator */
#define GEMM_MXF8_NUM_VARIANTS 5

/* D = act(A * B^T with block scales + bias), as above.
 *   A, B:        FP8 codes, M x K and N x K, 16-byte aligned (device memory).
 *   SFA, SFB:    tiled scales of A and B (gemm_mxf8_scale_bytes(M, K), (N, K) bytes),
 *                16-byte aligned.
 *   D:           M x N of out_dtype (GEMM_F16_DTYPE_F16 or _BF16), 16-byte aligned.
 *   fmt_a/fmt_b: GEMM_MXF8_E4M3 or GEMM_MXF8_E5M2.
 *   bias:        N elements of out_dtype, 16-byte aligned, or NULL; activation GEMM_F16_ACT_*.
 *   variant:     GEMM_MXF8_VARIANT_*; workspace/workspace_bytes as for gemm_f16_nt_ex (NULL/0:
 *                data-parallel schedule).
 * Errors: GEMM_F16_ERR_INVALID_ARG for a null pointer, a negative or too large size or an
 * unknown format, dtype, activation or variant; GEMM_F16_ERR_UNSUPPORTED when K is not a
 * multiple of 32, N not a multiple of 8, or a pointer is misaligned.  M == 0 or N == 0 does
 * nothing; K == 0 writes zeros (not with a bias or activation). */
int gemm_mxf8_nt(const void* A, const void* B, const void* SFA, const void* SFB, void* D,
                 int64_t M, int64_t N, int64_t K, int fmt_a, int fmt_b, int out_dtype,
                 const void* bias, int activation, int variant, void* workspace,
                 size_t workspace_bytes, cudaStream_t stream);

/* Workspace bytes for the stream-K tail of gemm_mxf8_nt with this shape and variant (0 when
 * the shape gets no tail). */
int gemm_mxf8_workspace_bytes(int64_t M, int64_t N, int64_t K, int variant, size_t* bytes);

/* The variant GEMM_MXF8_VARIANT_AUTO picks for this shape on a device with num_sms SMs. */
int gemm_mxf8_choose_variant(int64_t M, int64_t N, int64_t K, int num_sms);

/* Bytes of a tiled scale buffer for a rows x K operand; -1 if rows < 0 or K is not a
 * non-negative multiple of 32. */
int64_t gemm_mxf8_scale_bytes(int64_t rows, int64_t K);

/* Row-major scales (rows x K/32 bytes at src, device memory) -> the tiled layout at dst
 * (gemm_mxf8_scale_bytes(rows, K) bytes, device memory, not overlapping src), padding bytes set
 * to 127.  Asynchronous on `stream`. */
int gemm_mxf8_pack_scales(const void* src, void* dst, int64_t rows, int64_t K,
                          cudaStream_t stream);

/* Host-side encoders (no GPU needed): the instruction descriptor of the block-scaled MMA with
 * scale-factor IDs 0, the tiled-layout byte offset of scale (row, k_block) for a given K (-1 if
 * out of range), and the shared-memory descriptor of a 512-byte scale chunk. */
uint32_t gemm_mxf8_idesc(uint32_t M, uint32_t N, uint32_t fmt_a, uint32_t fmt_b);
int64_t gemm_mxf8_sf_offset(int64_t row, int64_t k_block, int64_t K);
uint64_t gemm_mxf8_sf_desc(uint32_t smem_addr);
int gemm_mxf8_get_variant_info(int variant, gemm_f16_variant_info* out);

#ifdef __cplusplus
}
#endif

#endif /* GEMM_F16_H */
