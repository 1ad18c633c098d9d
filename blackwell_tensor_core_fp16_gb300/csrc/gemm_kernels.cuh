// GEMM kernels for sm_103a: D = A * B^T with A (M x K) and B (N x K) fp16 row-major,
// fp32 accumulation in Tensor Memory, D (M x N) fp16 row-major.
//
// Two kernels:
//
//  * gemm_tile_kernel<BN>: one 128 x BN output tile per CTA (BN = 16 .. 128) on a 2-D grid, 4
//    warps, two shared-memory stages.  Thread 0 issues the TMA loads of a 64-wide K chunk a chunk
//    ahead, waits for them, issues four K=16 tcgen05.mma and commits them; then every warp reads
//    its 32 TMEM lanes, converts and stores its rows directly.  This is the protocol of Steps
//    2-4 on the page "TIRx 与高性能GEMM (上)" (a K loop whose first MMA overwrites the
//    accumulator, mbarrier phases flipped on every use, TMA loads completing on a
//    transaction-count barrier) with one load in flight behind the MMAs.  With a narrow BN it
//    is the fast path for problems of a few tiles, and the cross-check for the persistent kernel.
//
//  * gemm_ws_kernel<CtaGroup, BlockN, Stages>: the persistent, warp-specialised kernel.
//      warp 0      TMA producer: fills a ring of `Stages` shared-memory stages (A 128x64 and
//                  B (BlockN/CtaGroup)x64 per CTA, 128-byte swizzle), one "full" barrier per
//                  stage with an expected byte count, waiting on the stage's "empty" barrier.
//      warp 1      MMA issuer (one thread; in a CTA pair only the even CTA issues): four
//                  tcgen05.mma per stage into one of two TMEM accumulators, tcgen05.commit to
//                  the stage's "empty" barrier, and after the tile's last K chunk to the
//                  accumulator's "tmem_full" barrier.  Also allocates and frees TMEM.
//      warps 2-5   epilogue warpgroup: waits on "tmem_full", reads its TMEM lanes with
//                  tcgen05.ld 32x32b, frees the accumulator for the next tile ("tmem_empty"),
//                  converts fp32 -> fp16 with round-to-nearest-even, writes 128x64 swizzled
//                  sub-tiles to shared memory and stores them with TMA (double-buffered).
//    Tiles come from a static persistent schedule (tile = cluster id + i * clusters) in the
//    grouped order of tile_coord().  Ring and accumulator positions are counted across tiles,
//    so any K works.  Two accumulators let the epilogue of tile i overlap the MMAs of tile i+1.
//    With CtaGroup == 2, a cluster of two CTAs computes a 256 x BlockN tile with
//    tcgen05.mma.cta_group::2 (M = 256): each CTA loads its own 128 rows of A and its own half
//    of the BlockN rows of B, both CTAs' loads complete on the even CTA's "full" barrier, and
//    the MMA commit signals both CTAs.  No operand is shared, so no load is multicast.  The
//    last partial wave may run as half-width items (two per tile, N = BlockN / 2), and the
//    stream-K tail, when turned on, splits its tiles by k-blocks.
//
// Tails: TMA loads fill elements outside [0,M)x[0,K) and [0,N)x[0,K) with zeros, so partial K
// chunks add nothing and partial M/N tiles compute zeros in the padding; TMA stores and the
// direct stores of gemm_tile_kernel never write outside [0,M)x[0,N).
//
// Every wait is bounded.  A wait that runs out sets a bit in gemm_f16_status_word and the
// CTA's abort flag (so the CTA's other roles stop waiting too), the role waits (bounded) for the
// asynchronous work it issued, and the CTA frees its TMEM and exits.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_fp16.h>

#include "desc.h"
#include "ptx.cuh"

namespace gf16 {

// Debug flags of a launch (testing the failure path without faulting anything).
// kDebugNoLoads: the producer issues no copies and arms no barrier, so the first wait on a
// "full" barrier can only run out; nothing asynchronous is ever in flight.
constexpr uint32_t kDebugNoLoads = 1u;

// Bits reported through gemm_f16_status_word (read and cleared by the host).
constexpr uint32_t kStatusProducerTimeout = 1u;
constexpr uint32_t kStatusMmaTimeout = 2u;
constexpr uint32_t kStatusEpilogueTimeout = 4u;
constexpr uint32_t kStatusDrainTimeout = 8u;

__device__ uint32_t gemm_f16_status_word;

__device__ __forceinline__ void report(uint32_t bits, volatile uint32_t* abort_flag)
{
    *abort_flag = 1u;
    atomicOr(&gemm_f16_status_word, bits);
}

// Tiles a persistent unit (CTA or CTA pair) `c` of `units` processes: c, c + units, ...
__device__ __forceinline__ uint32_t tiles_of(uint32_t c, uint32_t units, uint32_t num_tiles)
{
    return c < num_tiles ? (num_tiles - c + units - 1u) / units : 0u;
}

constexpr uint32_t kBlockM = 128;  // rows of A (and D) per CTA
constexpr uint32_t kMaxContrib = 4;  // most stream-K pieces one tile is split into

// Stream-K workspace: a header of kSkHeaderBytes, then one slot of fp32 partial sums per unit
// and CTA.  The header must be zero when a workspace is first used; launches keep it so:
//   word 0   which of the two flag regions the current launch uses (0 or 1);
//   word 1   CTAs of the current launch that have finished (the last flips word 0 and clears
//            this count, so the next launch uses the other region);
//   words kSkFlagBase ..  flag region 0, then flag region 1, kSkFlagWords words each.  Flag
//            (tail tile r, contributor j, CTA rank) is 1 once that contributor's partial sums
//            are in its slot.  Each launch clears the region it does not use, so the next
//            launch finds its region zero, even after a launch that gave up a wait.
constexpr uint32_t kSkHeaderBytes = 8192;
constexpr uint32_t kSkFlagBase = 64;
constexpr uint32_t kSkFlagWords = (kSkHeaderBytes / 4u - kSkFlagBase) / 2u;
constexpr uint32_t kBlockK = 64;   // one 128-byte swizzle row of fp16
constexpr uint32_t kUmmaK = 16;    // K per tcgen05.mma of kind::f16

// ==============================================================================================
// gemm_tile_kernel: one 128 x kBN tile per CTA (kBN = 16 .. 128), a two-stage K loop run by one
// thread (the load of k-block kb + 1 overlaps the MMAs of k-block kb), the epilogue stores from
// registers.  For problems of a few tiles, where a launch's fixed costs dominate: a narrow kBN
// spreads a small D over more SMs, each loading and storing less.
// ==============================================================================================
template <uint32_t kBN>
struct TileCfg {
    static_assert(kBN >= 16 && kBN <= 128 && kBN % 16 == 0, "N of a kind::f16 MMA with M = 128");
    static constexpr uint32_t BN = kBN;
    static constexpr uint32_t A_BYTES = kBlockM * kBlockK * 2;  // 16384
    static constexpr uint32_t B_BYTES = BN * kBlockK * 2;       // 2048 .. 16384
    static constexpr uint32_t STAGE_TX = A_BYTES + B_BYTES;
    static constexpr uint32_t STAGE_BYTES = (STAGE_TX + 1023u) & ~1023u;
    static constexpr uint32_t STAGES = 2;
    static constexpr uint32_t OFF_BAR = STAGES * STAGE_BYTES;   // tma x2, mma, drain
    static constexpr uint32_t OFF_SLOT = OFF_BAR + 4 * 8;
    static constexpr uint32_t OFF_ABORT = OFF_SLOT + 4;
    static constexpr uint32_t SMEM_ALLOC = OFF_ABORT + 4 + 1024;
    static constexpr uint32_t TMEM_COLS = BN < 32 ? 32 : BN;   // a power of two >= 32
    static constexpr uint32_t LD_CHUNKS = (BN + 31) / 32;     // 32-column TMEM loads
    static constexpr uint32_t THREADS = 128;
};

template <uint32_t kBN>
__global__ void __launch_bounds__(128, 1)
    gemm_tile_kernel(const __grid_constant__ CUtensorMap tmap_a,
                     const __grid_constant__ CUtensorMap tmap_b, uint16_t* __restrict__ D,
                     uint32_t M, uint32_t N, uint32_t num_k_blocks, uint64_t timeout_ns,
                     uint32_t debug_flags)
{
    using C = TileCfg<kBN>;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t* base_ptr = smem_raw + (base - raw);
    const auto stage_a = [&](uint32_t s) { return base + s * C::STAGE_BYTES; };
    const auto stage_b = [&](uint32_t s) { return base + s * C::STAGE_BYTES + C::A_BYTES; };
    const uint32_t bar0 = base + C::OFF_BAR;
    const auto tma_bar = [&](uint32_t s) { return bar0 + 8u * s; };
    const uint32_t mma_bar = bar0 + 16;
    const uint32_t drain_bar = bar0 + 24;
    volatile uint32_t* slot_ptr = reinterpret_cast<volatile uint32_t*>(base_ptr + C::OFF_SLOT);
    volatile uint32_t* abort_flag = reinterpret_cast<volatile uint32_t*>(base_ptr + C::OFF_ABORT);

    const uint32_t warp = threadIdx.x >> 5;
    const uint32_t lane = threadIdx.x & 31u;
    const int32_t m0 = static_cast<int32_t>(blockIdx.y * kBlockM);
    const int32_t n0 = static_cast<int32_t>(blockIdx.x * C::BN);
    constexpr uint32_t idesc = make_idesc_f16(kBlockM, C::BN, 0);

    if (threadIdx.x == 0) {
        prefetch_tensormap(&tmap_a);
        prefetch_tensormap(&tmap_b);
        mbar_init(tma_bar(0), 1);
        mbar_init(tma_bar(1), 1);
        mbar_init(mma_bar, 1);
        mbar_init(drain_bar, 1);
        *abort_flag = 0u;
        fence_mbarrier_init();
    }
    __syncwarp();
    if (warp == 0) tmem_alloc<1>(smem_u32(const_cast<uint32_t*>(slot_ptr)), C::TMEM_COLS);
    tcgen05_fence_before();
    __syncthreads();
    tcgen05_fence_after();
    const uint32_t tmem_base = *slot_ptr;
    // As in the persistent kernels: the set-up above may overlap the end of the previous kernel
    // on the stream; global memory (A and B may be its output, D its input) waits for it.
    grid_dep_launch();
    grid_dep_wait();

    if (threadIdx.x == 0) {
        const bool loads = !(debug_flags & kDebugNoLoads);
        uint32_t loaded = 0, landed = 0;   // k-blocks whose loads were issued / waited for
        const auto load = [&](uint32_t kb) {
            const uint32_t s = kb & 1u;
            const int32_t k0 = static_cast<int32_t>(kb * kBlockK);
            mbar_arrive_expect_tx(tma_bar(s), C::STAGE_TX);
            tma_load_2d(stage_a(s), &tmap_a, tma_bar(s), k0, m0);
            tma_load_2d(stage_b(s), &tmap_b, tma_bar(s), k0, n0);
            ++loaded;
        };
        bool ok = true;
        bool issued_mma = false;
        // Phase j of mma_bar completes when the MMAs of k-block j are done.  A parity names one
        // phase only while at most one phase is pending, so each k-block's MMAs are committed
        // only after the previous k-block's are done (which also frees that k-block's stage for
        // the next load), and the phases are waited for in order.
        uint32_t mma_done = 0;
        const auto wait_mma = [&](uint32_t upto) {   // phases mma_done .. upto - 1
            for (; mma_done < upto; ++mma_done)
                if (!mbar_wait(mma_bar, mma_done & 1u, abort_flag, timeout_ns)) return false;
            return true;
        };
        if (loads) load(0);
        for (uint32_t kb = 0; kb < num_k_blocks; ++kb) {
            const uint32_t s = kb & 1u;
            if (!wait_mma(kb)) {
                report(kStatusMmaTimeout, abort_flag);
                ok = false;
                break;
            }
            // the other stage was last read by the MMAs of k-block kb - 1, now done
            if (kb + 1 < num_k_blocks && loads) load(kb + 1);
            if (!mbar_wait(tma_bar(s), (kb >> 1) & 1u, abort_flag, timeout_ns)) {
                report(kStatusProducerTimeout, abort_flag);
                ok = false;
                break;
            }
            ++landed;
            tcgen05_fence_after();
            const uint64_t ad = make_smem_desc_sw128(stage_a(s), 1024);
            const uint64_t bd = make_smem_desc_sw128(stage_b(s), 1024);
#pragma unroll
            for (uint32_t k = 0; k < kBlockK / kUmmaK; ++k)
                mma_f16<1>(tmem_base, ad + 2ull * k, bd + 2ull * k, idesc, (kb | k) != 0u);
            mma_commit(mma_bar);   // phase kb of mma_bar: the MMAs of k-block kb are done
            issued_mma = true;
        }
        if (ok && !wait_mma(num_k_blocks)) {
            report(kStatusMmaTimeout, abort_flag);
            ok = false;
        }
        if (!ok) {
            // Let every MMA this thread issued finish before TMEM is freed, and every load
            // issued land before the CTA exits (bounded waits that ignore the abort flag).
            if (issued_mma) {
                mma_commit(drain_bar);
                if (!mbar_wait(drain_bar, 0, nullptr, timeout_ns))
                    atomicOr(&gemm_f16_status_word, kStatusDrainTimeout);
            }
            for (uint32_t kb = landed; kb < loaded; ++kb)
                if (!mbar_wait(tma_bar(kb & 1u), (kb >> 1) & 1u, nullptr, timeout_ns))
                    atomicOr(&gemm_f16_status_word, kStatusDrainTimeout);
        }
    }
    __syncwarp();
    tcgen05_fence_before();
    __syncthreads();
    tcgen05_fence_after();

    if (*abort_flag == 0u) {
        // TMEM lane = row of the tile; warp w may read lanes 32w .. 32w + 31.  All the 32-column
        // loads are in flight before one wait (past column BN they read unused columns).
        const uint32_t row = warp * 32u + lane;
        const uint32_t grow = static_cast<uint32_t>(m0) + row;
        uint32_t v[C::LD_CHUNKS][32];
#pragma unroll
        for (uint32_t c = 0; c < C::LD_CHUNKS; ++c)
            tmem_ld_32x32b_x32(tmem_base + ((warp * 32u) << 16), v[c], static_cast<int>(c * 32u));
        tmem_ld_wait();
        if (grow < M) {
#pragma unroll
            for (uint32_t c = 0; c < C::LD_CHUNKS; ++c) {
                uint32_t p[16];
#pragma unroll
                for (int i = 0; i < 16; ++i) p[i] = pack_f16x2_rn(v[c][2 * i], v[c][2 * i + 1]);
#pragma unroll
                for (uint32_t q = 0; q < 4; ++q) {
                    const uint32_t col = static_cast<uint32_t>(n0) + c * 32u + q * 8u;
                    // N is a multiple of 8: a vector is all in or all out
                    if (c * 32u + q * 8u < C::BN && col < N)
                        st_global_v4(D + static_cast<uint64_t>(grow) * N + col, p[4 * q],
                                     p[4 * q + 1], p[4 * q + 2], p[4 * q + 3]);
                }
            }
        }
    }
    tcgen05_fence_before();
    __syncthreads();
    if (warp == 0) {
        tcgen05_fence_after();
        tmem_dealloc<1>(tmem_base, C::TMEM_COLS);
    }
}

// ==============================================================================================
// The fused epilogue of a linear layer: y = act(x + bias[column]) on the fp32 accumulator,
// before the single rounding to the output type.  act: 0 none, 1 ReLU, 2 GELU (exact form,
// x * Phi(x) = x/2 * erfc(-x / sqrt 2)).
// ==============================================================================================
constexpr uint32_t kActNone = 0, kActRelu = 1, kActGelu = 2;

// GELU in its exact form x Phi(x), Phi(x) = erfc(-x / sqrt 2) / 2, with erfc from the Chebyshev
// fit of Press, Teukolsky, Vetterling and Flannery, Numerical Recipes (2nd ed.), section 6.2:
// for z >= 0, erfc(z) = t exp(-z^2 + P(t)) with t = 1 / (1 + z/2) and P a degree-9 polynomial,
// fractional error below 1.2e-7 in exact arithmetic.  Phi(x) is then 1 - erfc(|x| / sqrt 2) / 2
// for x >= 0 and erfc(|x| / sqrt 2) / 2 below, so the small tail is never the difference of two
// near-equal numbers.  Branch-free, one reciprocal and one exponential per value; evaluated in
// fp32 it stays within 2e-7 (plus one fp32 rounding of the result) of the exact GELU for
// |x| <= 10; the output is then rounded to a 16-bit type.
__device__ __forceinline__ float gelu_exact(float x)
{
    const float z = fabsf(x) * 0.70710678118654752f;
    const float t = __fdividef(1.f, fmaf(0.5f, z, 1.f));
    float p = 0.17087277f;
    p = fmaf(p, t, -0.82215223f);
    p = fmaf(p, t, 1.48851587f);
    p = fmaf(p, t, -1.13520398f);
    p = fmaf(p, t, 0.27886807f);
    p = fmaf(p, t, -0.18628806f);
    p = fmaf(p, t, 0.09678418f);
    p = fmaf(p, t, 0.37409196f);
    p = fmaf(p, t, 1.00002368f);
    p = fmaf(p, t, -1.26551223f);
    const float e = t * expf(fmaf(-z, z, p));   // erfc(|x| / sqrt 2)
    return x * (x >= 0.f ? fmaf(-0.5f, e, 1.f) : 0.5f * e);
}

// GELU of eight values in one call.  Not inlined: every 64-column chunk the epilogue emits
// would otherwise carry 64 inlined copies (tens of KB of instructions per kernel, which the
// instruction cache does not hold); eight values per call keep eight independent chains in
// flight.  (Measured on the MLP shape, bf16 with bias: inlined, the GELU epilogue took the
// launch from 1.04 to 1.53 ms; eight per call, 1.13 ms; sixteen per call was slower again.)
struct F8 { float v[8]; };
__device__ __noinline__ F8 gelu8(F8 x)
{
#pragma unroll
    for (int i = 0; i < 8; ++i) x.v[i] = gelu_exact(x.v[i]);
    return x;
}

__device__ __forceinline__ float apply_act(float v, uint32_t act)
{
    if (act == kActRelu) return fmaxf(v, 0.f);
    if (act == kActGelu) return gelu_exact(v);
    return v;
}

// Widen a 16-bit element of the given type (fp16 or bf16) to fp32.
template <bool kBf16>
__device__ __forceinline__ float widen16(uint32_t h)
{
    if constexpr (kBf16) return __uint_as_float(h << 16);
    else return __half2float(__ushort_as_half(static_cast<unsigned short>(h)));
}

// 8 consecutive fp32 accumulators of columns col .. col+7 -> act(acc + bias).  `col` is a
// multiple of 8 and N % 8 == 0, so the 16-byte bias vector is all in or all out.
// kCall: GELU through the non-inlined gelu8 (false: inlined, for the one-accumulator epilogue,
// whose registers hold the whole packed tile and leave none for a call).
template <bool kBf16, bool kCall = true>
__device__ __forceinline__ void epilogue8(float (&v)[8], const uint16_t* bias, int32_t col,
                                          uint32_t N, uint32_t act)
{
    if (bias != nullptr && col < static_cast<int32_t>(N)) {
        const uint4 b = __ldg(reinterpret_cast<const uint4*>(bias + col));
        const uint32_t w[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            v[2 * i] += widen16<kBf16>(w[i] & 0xFFFFu);
            v[2 * i + 1] += widen16<kBf16>(w[i] >> 16);
        }
    }
    if (kCall && act == kActGelu) {
        F8 x;
#pragma unroll
        for (int i = 0; i < 8; ++i) x.v[i] = v[i];
        x = gelu8(x);
#pragma unroll
        for (int i = 0; i < 8; ++i) v[i] = x.v[i];
    } else if (act != kActNone) {
#pragma unroll
        for (int i = 0; i < 8; ++i) v[i] = apply_act(v[i], act);
    }
}

template <bool kBf16>
__device__ __forceinline__ uint32_t pack2(uint32_t lo_bits, uint32_t hi_bits)
{
    if constexpr (kBf16) return pack_bf16x2_rn(lo_bits, hi_bits);
    else return pack_f16x2_rn(lo_bits, hi_bits);
}

// ==============================================================================================
// gemm_ws_kernel: persistent, warp-specialised, TMEM double-buffered.
// ==============================================================================================
// kMx: block-scaled FP8 operands (E4M3/E5M2 with one E8M0 scale per 32 K elements) instead of
// fp16/bf16.  A stage still holds 128-byte rows (128 FP8 elements instead of 64 fp16), plus the
// stage's scale chunks (see mx_sf_offset): one for this CTA's 128 rows of A and SFB_CHUNKS for
// the tile's rows of B, which every CTA of a pair loads whole.  The MMA issuer copies them into
// a ring of tensor-memory columns after the two accumulators, one slot per stage.
// kAccBufs: tensor-memory accumulators (2: the epilogue of tile i overlaps the MMAs of tile
// i + 1; 1: a 256-column accumulator leaves room for the block scales, and the epilogue reads it
// out into registers before it stores, so the MMAs wait only for that read).
// kDBufs: shared-memory staging buffers of the TMA-store epilogue (2: a sub-tile is written
// while the previous one is still being stored; 1 frees 16 KB for another pipeline stage where
// the stores are off the critical path, as after a single accumulator has been read out).
template <int kCtaGroup, int kBlockN, int kStages, bool kTmaStore = true, bool kMx = false,
          int kAccBufs = 2, int kDBufs = 2>
struct WsCfg {
    static_assert(kAccBufs == 1 || kAccBufs == 2, "one or two accumulators");
    static_assert(kDBufs == 1 || kDBufs == 2, "one or two staging buffers");
    static constexpr uint32_t ACC_BUFS = kAccBufs;
    static constexpr uint32_t D_BUFS = kDBufs;
    static_assert(kCtaGroup == 1 || kCtaGroup == 2, "a CTA or a CTA pair");
    static_assert(kBlockN % 64 == 0 && kBlockN >= 64 && kBlockN <= 256, "N tile");
    static constexpr uint32_t BN = kBlockN;
    static constexpr uint32_t MMA_M = kBlockM * kCtaGroup;
    static constexpr uint32_t B_ROWS = kBlockN / kCtaGroup;  // rows of B each CTA loads
    static constexpr uint32_t ELEM_BYTES = kMx ? 1u : 2u;
    static constexpr uint32_t BLOCK_K = 128u / ELEM_BYTES;   // elements in a 128-byte row
    static constexpr uint32_t A_BYTES = kBlockM * 128u;
    static constexpr uint32_t B_BYTES = B_ROWS * 128u;
    static constexpr uint32_t SFB_CHUNKS = kMx ? (kBlockN % 128 == 0 ? kBlockN / 128 : kBlockN / 128 + 1) : 0u;
    static constexpr uint32_t SF_BYTES = kMx ? 512u * (1u + SFB_CHUNKS) : 0u;
    static constexpr uint32_t SF_COLS = kMx ? 4u * (1u + SFB_CHUNKS) : 0u;  // TMEM cols per stage
    static constexpr uint32_t TMEM_SF = kAccBufs * kBlockN;    // first scale-factor column
    // Bytes that complete on the issuing CTA's "full" barrier per stage (both CTAs' loads).
    static constexpr uint32_t STAGE_TX = (A_BYTES + B_BYTES + SF_BYTES) * kCtaGroup;
    // a half-width item (the first B_ROWS / 2 rows of each CTA's B stage; no scales)
    static constexpr uint32_t STAGE_TX_HALF = (A_BYTES + B_BYTES / 2) * kCtaGroup;
    static constexpr uint32_t D_COLS = 64;                   // one 128-byte swizzle row of fp16
    static constexpr uint32_t D_BYTES = kBlockM * D_COLS * 2;
    // accumulators (+ scales), rounded up to the power of two tcgen05.alloc takes
    static constexpr uint32_t TMEM_COLS =
        kMx ? 512u : (kAccBufs * kBlockN <= 128u ? 128u : kAccBufs * kBlockN <= 256u ? 256u : 512u);
    static_assert((TMEM_COLS & (TMEM_COLS - 1)) == 0 && TMEM_COLS <= 512, "TMEM columns");
    static_assert(!kMx || TMEM_SF + kStages * SF_COLS <= TMEM_COLS, "TMEM scale-factor ring");
    static constexpr uint32_t OFF_A = 0;
    static constexpr uint32_t OFF_B = OFF_A + kStages * A_BYTES;
    static constexpr uint32_t OFF_SF = OFF_B + kStages * B_BYTES;
    // the swizzled D staging buffers start on a 1024-byte boundary
    static constexpr uint32_t OFF_D = (OFF_SF + kStages * SF_BYTES + 1023u) & ~1023u;
    // Two staging buffers for the TMA-store epilogue; none when the epilogue stores directly.
    static constexpr uint32_t OFF_BAR = OFF_D + (kTmaStore ? kDBufs * D_BYTES : 0);
    static constexpr uint32_t NUM_BARS = 2 * kStages + 6;  // full, empty, tfull x2, tempty x2, drain, pair
    static constexpr uint32_t OFF_SLOT = OFF_BAR + NUM_BARS * 8;
    static constexpr uint32_t OFF_ABORT = OFF_SLOT + 4;
    static constexpr uint32_t OFF_EPI_WORD = OFF_ABORT + 4;      // epilogue broadcast word
    static constexpr uint32_t SMEM_ALLOC = OFF_EPI_WORD + 4 + 1024;  // + slack to align the base
    // Stream-K workspace: one fp32 partial accumulator per (unit, piece, CTA of the pair).
    static constexpr uint32_t PART_FLOATS = kBlockM * kBlockN;
    static_assert(SMEM_ALLOC <= 232448, "shared memory per CTA");
    static constexpr uint32_t THREADS = 192;
    static constexpr uint32_t EPI_THREADS = 128;
};

// kBf16: bf16 operands and output (fp16 otherwise); with kMx it selects the output type only.
template <int kCtaGroup, int kBlockN, int kStages, bool kTmaStore, bool kBf16 = false,
          bool kMx = false, int kAccBufs = 2, int kDBufs = 2>
__global__ void __launch_bounds__(192, 1)
    gemm_ws_kernel(const __grid_constant__ CUtensorMap tmap_a,
                   const __grid_constant__ CUtensorMap tmap_b,
                   const __grid_constant__ CUtensorMap tmap_d, uint16_t* __restrict__ Dptr,
                   uint32_t M, uint32_t N,
                   uint32_t num_m_blocks, uint32_t num_n_blocks, uint32_t num_k_blocks,
                   uint32_t group_m, uint64_t timeout_ns, uint32_t l2_hints,
                   float* __restrict__ ws_part, uint32_t* __restrict__ ws_hdr,
                   uint32_t sk_tiles, uint32_t sk_units, const uint16_t* __restrict__ bias,
                   uint32_t act, uint32_t debug_flags,
                   const __grid_constant__ CUtensorMap tmap_sfa,
                   const __grid_constant__ CUtensorMap tmap_sfb, uint32_t mx_idesc,
                   const __grid_constant__ CUtensorMap tmap_b_half, uint32_t half_tiles)
{
    using C = WsCfg<kCtaGroup, kBlockN, kStages, kTmaStore, kMx, kAccBufs, kDBufs>;
    constexpr bool kPair = (kCtaGroup == 2);
    constexpr uint32_t idesc = make_idesc_f16(C::MMA_M, C::BN, kBf16 ? 1u : 0u);
    constexpr uint32_t idesc_half = make_idesc_f16(C::MMA_M, C::BN / 2, kBf16 ? 1u : 0u);
    // Half-width tail items exist only on the 16-bit path and when half a tile is a whole number
    // of the epilogue's 64-column chunks (the host passes half_tiles = 0 otherwise).
    constexpr bool kHalves = !kMx && (kBlockN / 2) % 64 == 0;
    const bool fused = bias != nullptr || act != kActNone;

    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t* base_ptr = smem_raw + (base - raw);
    const uint32_t sA = base + C::OFF_A;
    const uint32_t sB = base + C::OFF_B;
    const uint32_t sSF = base + C::OFF_SF;
    const uint32_t sD = base + C::OFF_D;
    const uint32_t bar0 = base + C::OFF_BAR;
    const auto full_bar = [&](uint32_t s) { return bar0 + 8u * s; };
    const auto empty_bar = [&](uint32_t s) { return bar0 + 8u * (kStages + s); };
    const auto tfull_bar = [&](uint32_t b) { return bar0 + 8u * (2u * kStages + b); };
    const auto tempty_bar = [&](uint32_t b) { return bar0 + 8u * (2u * kStages + 2u + b); };
    const uint32_t drain_bar = bar0 + 8u * (2u * kStages + 4u);
    const uint32_t pair_bar = bar0 + 8u * (2u * kStages + 5u);   // teardown rendezvous of a pair
    volatile uint32_t* slot_ptr = reinterpret_cast<volatile uint32_t*>(base_ptr + C::OFF_SLOT);
    volatile uint32_t* abort_flag = reinterpret_cast<volatile uint32_t*>(base_ptr + C::OFF_ABORT);

    const uint32_t warp = threadIdx.x >> 5;
    const uint32_t lane = threadIdx.x & 31u;
    const uint32_t rank = kPair ? cluster_ctarank() : 0u;
    const uint32_t cid = kPair ? cluster_id_x() : blockIdx.x;
    const uint32_t ncl = kPair ? num_clusters_x() : gridDim.x;
    const uint32_t num_tiles = num_m_blocks * num_n_blocks;
    // Work of this unit: its data-parallel tiles, then (sk_tiles > 0) its stream-K pieces.
    const WorkSplit split{num_tiles, ncl, num_k_blocks, sk_tiles, sk_units, half_tiles};
    const uint32_t n_items = items_of(split, cid);
    const uint32_t total = iterations_of(split, cid);

    // ---- set-up: barriers, TMEM ----------------------------------------------------------
    if (threadIdx.x == 0) {
        prefetch_tensormap(&tmap_a);
        prefetch_tensormap(&tmap_b);
        prefetch_tensormap(&tmap_d);
        if (half_tiles != 0u) prefetch_tensormap(&tmap_b_half);
        if constexpr (kMx) {
            prefetch_tensormap(&tmap_sfa);
            prefetch_tensormap(&tmap_sfb);
        }
        for (uint32_t s = 0; s < kStages; ++s) {
            mbar_init(full_bar(s), 1);
            mbar_init(empty_bar(s), 1);
        }
        for (uint32_t b = 0; b < 2; ++b) {
            mbar_init(tfull_bar(b), 1);
            mbar_init(tempty_bar(b), 4u * kCtaGroup);  // one arrival per epilogue warp per CTA
        }
        mbar_init(drain_bar, 1);
        mbar_init(pair_bar, 1);
        *abort_flag = 0u;
        fence_mbarrier_init();
    }
    __syncwarp();
    if (warp == 1) {
        tmem_alloc<kCtaGroup>(smem_u32(const_cast<uint32_t*>(slot_ptr)), C::TMEM_COLS);
        tmem_relinquish<kCtaGroup>();
    }
    tcgen05_fence_before();
    // The barriers and the TMEM address become visible to the CTA (to the pair: at the cluster
    // barrier, whose latency, about 1000 cycles on GB300, each role overlaps with its own
    // register-only set-up before it waits).
    if constexpr (kPair) cluster_arrive(); else __syncthreads();
    // Everything so far touches only shared memory, tensor memory and the kernel parameters, so
    // it may overlap the end of the previous kernel on the stream: let the next GEMM begin its
    // own set-up as SMs free up.  The roles that touch global memory (the producer's loads of
    // A and B, which may be the previous kernel's output; the epilogue's stores of D, which it
    // may read) wait for the previous kernel first; the MMA issuer needs no wait.
    grid_dep_launch();
    uint32_t tmem_base = 0;
    const auto setup_done = [&]() {
        if constexpr (kPair) cluster_wait();
        tcgen05_fence_after();
        tmem_base = *slot_ptr;
    };

    if (warp == 0) {
        // ---- TMA producer ------------------------------------------------------------------
        // The whole warp runs the loop, so every value it computes is warp-uniform; the waits'
        // outcome is agreed by a vote, and one elected lane issues the copies.
        const bool leader = elect_one_sync();
        // L2 priorities of A and B loads (bits 1:0 and 3:2 of l2_hints; 0 = normal).
        const uint64_t pol_a = make_l2_policy(l2_hints & 3u);
        const uint64_t pol_b = make_l2_policy((l2_hints >> 2) & 3u);
        uint32_t it = 0;
        bool ok = true;
        uint32_t item = 0;
        WorkItem wi = work_item(split, cid, 0);
        uint32_t kb = wi.kb0;
        int32_t m0 = 0, n0 = 0, sf_rb_b = 0;
        const auto tile_origin = [&]() {
            const TileCoord tc = tile_coord(wi.tile, num_m_blocks, num_n_blocks, group_m);
            m0 = static_cast<int32_t>(tc.m_blk * C::MMA_M + rank * kBlockM);
            // a half-width item: its columns start half a tile in for the second half, and each
            // CTA loads half as many rows of B
            n0 = (!kHalves || wi.half == 0u)
                     ? static_cast<int32_t>(tc.n_blk * C::BN + rank * C::B_ROWS)
                     : static_cast<int32_t>(tc.n_blk * C::BN + (wi.half - 1u) * (C::BN / 2u) +
                                            rank * (C::B_ROWS / 2u));
            // the 128-row group of B's scales that holds the tile's first row
            sf_rb_b = static_cast<int32_t>(tc.n_blk * C::BN / 128u);
        };
        tile_origin();
        const uint32_t produce = (debug_flags & kDebugNoLoads) ? 0u : total;
        setup_done();
        grid_dep_wait();
        for (; it < produce; ++it) {
            if (kb == wi.kb0 && it != 0) tile_origin();
            const RingPos p = ring_pos(it, kStages);
            const bool w = mbar_wait<kPair>(empty_bar(p.stage), p.parity ^ 1u, abort_flag,
                                            timeout_ns);
            if (!__all_sync(0xffffffffu, w)) {
                if (leader) report(kStatusProducerTimeout, abort_flag);
                ok = false;
                break;
            }
            if (leader) {
                const int32_t k0 = static_cast<int32_t>(kb * C::BLOCK_K);
                const uint32_t dA = sA + p.stage * C::A_BYTES;
                const uint32_t dB = sB + p.stage * C::B_BYTES;
                const uint32_t dS = sSF + p.stage * C::SF_BYTES;
                const bool hw = kHalves && wi.half != 0u;   // a half-width item
                if constexpr (!kPair) {
                    mbar_arrive_expect_tx(full_bar(p.stage), hw ? C::STAGE_TX_HALF : C::STAGE_TX);
                    tma_load_2d_hint(dA, &tmap_a, full_bar(p.stage), k0, m0, pol_a);
                    tma_load_2d_hint(dB, hw ? &tmap_b_half : &tmap_b, full_bar(p.stage), k0, n0,
                                     pol_b);
                    if constexpr (kMx) {
                        // scale chunks (K-block group kb): A's row group, then B's groups
                        tma_load_3d(dS, &tmap_sfa, full_bar(p.stage), 0, static_cast<int32_t>(kb),
                                    m0 / 128);
                        tma_load_3d(dS + 512u, &tmap_sfb, full_bar(p.stage), 0,
                                    static_cast<int32_t>(kb), sf_rb_b);
                    }
                } else {
                    if (rank == 0)
                        mbar_arrive_expect_tx(full_bar(p.stage),
                                              hw ? C::STAGE_TX_HALF : C::STAGE_TX);
                    const uint32_t fb = mapa_shared(full_bar(p.stage), 0);
                    tma_load_2d_pair_hint(dA, &tmap_a, fb, k0, m0, pol_a);
                    tma_load_2d_pair_hint(dB, hw ? &tmap_b_half : &tmap_b, fb, k0, n0, pol_b);
                    if constexpr (kMx) {
                        tma_load_3d_pair(dS, &tmap_sfa, fb, 0, static_cast<int32_t>(kb), m0 / 128);
                        tma_load_3d_pair(dS + 512u, &tmap_sfb, fb, 0, static_cast<int32_t>(kb),
                                         sf_rb_b);
                    }
                }
            }
            __syncwarp();
            if (++kb == wi.kb1 && ++item < n_items) {
                wi = work_item(split, cid, item);
                kb = wi.kb0;
            }
        }
        // Every stage must be released by the MMAs before this CTA may exit: the last commits
        // still arrive on the "empty" barriers (in a pair, from the other CTA).  Iteration j is
        // released when phase j / Stages of its stage's barrier completes.
        const uint32_t first = it > kStages ? it - kStages : 0u;
        if (ok) {
            for (uint32_t j = first; j < it; ++j) {
                const RingPos p = ring_pos(j, kStages);
                const bool w = mbar_wait<kPair>(empty_bar(p.stage), p.parity, abort_flag,
                                                timeout_ns);
                if (!__all_sync(0xffffffffu, w)) {
                    if (leader) report(kStatusDrainTimeout, abort_flag);
                    break;
                }
            }
        } else if (rank == 0) {
            // After an abort: wait (bounded, ignoring the abort flag) for loads still in flight
            // into the ring, so none lands after this CTA has exited.
            for (uint32_t j = first; j < it; ++j) {
                const RingPos p = ring_pos(j, kStages);
                const bool w = mbar_wait<kPair>(full_bar(p.stage), p.parity, nullptr,
                                                timeout_ns / 8);
                if (!__all_sync(0xffffffffu, w)) break;
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        // ---- MMA issuer (the even CTA of a pair issues for both) ----------------------------
        // Warp-uniform loop as in the producer; one elected lane issues the MMAs and commits
        // (a commit tracks the MMAs its own thread issued, so it is always the same lane).
        setup_done();
        if (rank == 0) {
            const bool leader = elect_one_sync();
            uint32_t item = 0;
            WorkItem wi = work_item(split, cid, 0);
            uint32_t kb = wi.kb0;
            uint32_t acc = 0;
            uint32_t d_tmem = tmem_base;
            uint32_t sfb_shift = 0;
            bool ok = true;
            bool issued = false;
            for (uint32_t it = 0; it < total; ++it) {
                if (kb == wi.kb0) {
                    // A new tile: wait until the epilogue has drained accumulator acc % 2.
                    const uint32_t b = acc % C::ACC_BUFS;
                    const bool w = mbar_wait<kPair>(tempty_bar(b), ((acc / C::ACC_BUFS) & 1u) ^ 1u,
                                                    abort_flag, timeout_ns);
                    if (!__all_sync(0xffffffffu, w)) {
                        if (leader) report(kStatusMmaTimeout, abort_flag);
                        ok = false;
                        break;
                    }
                    tcgen05_fence_after();
                    d_tmem = tmem_base + b * C::BN;
                    if constexpr (kMx) {
                        // B's scales start at the tile's first row inside its first chunk.
                        const TileCoord tc =
                            tile_coord(wi.tile, num_m_blocks, num_n_blocks, group_m);
                        sfb_shift = ((tc.n_blk * C::BN) % 128u) / 32u;
                    }
                }
                const RingPos p = ring_pos(it, kStages);
                const bool w = mbar_wait<kPair>(full_bar(p.stage), p.parity, abort_flag,
                                                timeout_ns);
                if (!__all_sync(0xffffffffu, w)) {
                    if (leader) report(kStatusMmaTimeout, abort_flag);
                    ok = false;
                    break;
                }
                tcgen05_fence_after();
                const uint64_t ad = make_smem_desc_sw128(sA + p.stage * C::A_BYTES, 1024);
                const uint64_t bd = make_smem_desc_sw128(sB + p.stage * C::B_BYTES, 1024);
                if (leader) {
                    if constexpr (kMx) {
                        // This stage's scales -> its tensor-memory slot, then 4 MMAs of K = 32
                        // (one scale block each; the scale-factor ID picks the block's byte).
                        const uint32_t sf_col = tmem_base + C::TMEM_SF + p.stage * C::SF_COLS;
                        const uint32_t sS = sSF + p.stage * C::SF_BYTES;
#pragma unroll
                        for (uint32_t c = 0; c <= C::SFB_CHUNKS; ++c)
                            tmem_cp_32x128b_warpx4<kCtaGroup>(sf_col + 4u * c,
                                                              make_sf_desc(sS + 512u * c));
#pragma unroll
                        for (uint32_t k = 0; k < 4; ++k)
                            mma_mx<kCtaGroup>(d_tmem, ad + 2ull * k, bd + 2ull * k,
                                              idesc_mx_with_sf_id(mx_idesc, k), sf_col,
                                              sf_col + 4u + sfb_shift,
                                              ((kb - wi.kb0) | k) != 0u);
                    } else {
                        // a half-width item: N = BN / 2 from the first rows of each B stage
                        const uint32_t id = (kHalves && wi.half != 0u) ? idesc_half : idesc;
#pragma unroll
                        for (uint32_t k = 0; k < kBlockK / kUmmaK; ++k)
                            mma_f16<kCtaGroup>(d_tmem, ad + 2ull * k, bd + 2ull * k, id,
                                               ((kb - wi.kb0) | k) != 0u);
                    }
                    if constexpr (kPair) mma_commit_pair(empty_bar(p.stage), 0x3);
                    else mma_commit(empty_bar(p.stage));
                }
                __syncwarp();
                issued = true;
                if (++kb == wi.kb1) {
                    // Item done: the accumulator is ready for the epilogue once these MMAs are.
                    if (leader) {
                        if constexpr (kPair) mma_commit_pair(tfull_bar(acc % C::ACC_BUFS), 0x3);
                        else mma_commit(tfull_bar(acc % C::ACC_BUFS));
                    }
                    __syncwarp();
                    ++acc;
                    if (++item < n_items) {
                        wi = work_item(split, cid, item);
                        kb = wi.kb0;
                    }
                }
            }
            if (!ok && issued && leader) {
                // Let every MMA issued so far finish before TMEM is freed.
                if constexpr (kPair) mma_commit_pair(drain_bar, 0x1);
                else mma_commit(drain_bar);
                if (!mbar_wait<false>(drain_bar, 0, nullptr, timeout_ns))
                    atomicOr(&gemm_f16_status_word, kStatusDrainTimeout);
            }
            if constexpr (kPair) {
                // Both CTAs' epilogues hand each accumulator back with an arrival on this CTA's
                // barriers, the other CTA's from afar: wait for the last hand-backs, so that
                // none is still on its way when this CTA exits.
                for (uint32_t a = acc; ok && a < acc + C::ACC_BUFS; ++a) {
                    if (a < C::ACC_BUFS) continue;   // this buffer was never used
                    const bool w = mbar_wait<kPair>(tempty_bar(a % C::ACC_BUFS),
                                                    ((a / C::ACC_BUFS) & 1u) ^ 1u, abort_flag,
                                                    timeout_ns);
                    if (!__all_sync(0xffffffffu, w)) {
                        if (leader) report(kStatusMmaTimeout, abort_flag);
                        ok = false;
                    }
                }
            }
        }
        __syncwarp();
    } else {
        // ---- epilogue warpgroup ------------------------------------------------------------
        setup_done();
        grid_dep_wait();
        const uint32_t quad = warp & 3u;             // TMEM lanes 32*quad .. 32*quad + 31
        const uint32_t row = quad * 32u + lane;      // row of this CTA's 128-row slab
        const uint32_t et = threadIdx.x - 64u;       // 0 .. 127
        // Stream-K: this launch's flag region; the other one is cleared for the next launch.
        uint32_t* sk_flags = nullptr;
        if (sk_tiles != 0u) {
            const uint32_t region = __ldcg(ws_hdr) & 1u;
            sk_flags = ws_hdr + kSkFlagBase + region * kSkFlagWords;
            uint32_t* other = ws_hdr + kSkFlagBase + (region ^ 1u) * kSkFlagWords;
            for (uint32_t w = blockIdx.x * C::EPI_THREADS + et; w < kSkFlagWords;
                 w += gridDim.x * C::EPI_THREADS)
                other[w] = 0u;
        }
        const uint32_t lane_off = (quad * 32u) << 16;
        uint32_t sbuf = 0;
        // L2 priority of the D stores (bits 5:4 of l2_hints; 0 = normal)
        const uint64_t pol_d = make_l2_policy((l2_hints >> 4) & 3u);

        // Store 64 columns (32 packed f16x2 words) of this thread's row at column col0.
        const auto store_chunk = [&](const uint32_t (&p)[32], int32_t m0, int32_t col0) {
            if constexpr (kTmaStore) {
                // The store issued D_BUFS sub-tiles ago read this buffer; wait until it has.
                if (et == 0) bulk_wait_group_read<C::D_BUFS - 1>();
                __syncwarp();
                named_barrier_sync(1, C::EPI_THREADS);
                const uint32_t dbuf = sD + sbuf * C::D_BYTES;
#pragma unroll
                for (uint32_t j = 0; j < 8; ++j)
                    st_shared_v4(dbuf + sw128(row * 128u + j * 16u), p[4 * j], p[4 * j + 1],
                                 p[4 * j + 2], p[4 * j + 3]);
                fence_proxy_async_smem();
                named_barrier_sync(1, C::EPI_THREADS);
                if (et == 0) {
                    tma_store_2d_hint(&tmap_d, dbuf, col0, m0, pol_d);
                    bulk_commit_group();
                }
                __syncwarp();
                sbuf = (sbuf + 1u) % C::D_BUFS;
            } else {
                // Each thread writes its own row: 64 fp16 as 8 16-byte vectors; the L2 merges
                // the warp's 32 partial lines into full lines.
                const int32_t grow = m0 + static_cast<int32_t>(row);
                if (grow < static_cast<int32_t>(M)) {
                    uint16_t* drow = Dptr + static_cast<uint64_t>(grow) * N;
#pragma unroll
                    for (uint32_t j = 0; j < 8; ++j) {
                        const int32_t col = col0 + static_cast<int32_t>(8u * j);
                        if (col < static_cast<int32_t>(N))  // N % 8 == 0
                            st_global_v4(drow + col, p[4 * j], p[4 * j + 1], p[4 * j + 2],
                                         p[4 * j + 3]);
                    }
                }
            }
        };

        // A unit's partial sums live in its workspace slot in a layout where a warp's 32 rows
        // of one 16-byte column group are contiguous: float4 index ((chunk * 16 + j) * 128 + row).
        const auto part_of = [&](uint32_t unit) {
            return reinterpret_cast<float4*>(
                ws_part + (static_cast<uint64_t>(unit) * kCtaGroup + rank) * C::PART_FLOATS);
        };

        // Hand accumulator b back to the MMA issuer once this warp's loads of it are complete.
        const auto hand_back = [&](uint32_t b) {
            tcgen05_fence_before();
            __syncwarp();
            if (lane == 0) {
                if constexpr (kPair) mbar_arrive_remote(mapa_shared(tempty_bar(b), 0));
                else mbar_arrive_local(tempty_bar(b));
            }
            __syncwarp();
        };
        // Fused epilogue (if any), rounding and store of 64 fp32 columns (v0: the first 32).
        const auto emit64 = [&](uint32_t (&v0)[32], uint32_t (&v1)[32], int32_t m0, int32_t col0) {
            if (fused) {
#pragma unroll
                for (int g8 = 0; g8 < 4; ++g8) {
                    float f[8];
#pragma unroll
                    for (int i = 0; i < 8; ++i) f[i] = __uint_as_float(v0[8 * g8 + i]);
                    epilogue8<kBf16>(f, bias, col0 + 8 * g8, N, act);
#pragma unroll
                    for (int i = 0; i < 8; ++i) v0[8 * g8 + i] = __float_as_uint(f[i]);
                }
#pragma unroll
                for (int g8 = 0; g8 < 4; ++g8) {
                    float f[8];
#pragma unroll
                    for (int i = 0; i < 8; ++i) f[i] = __uint_as_float(v1[8 * g8 + i]);
                    epilogue8<kBf16>(f, bias, col0 + 32 + 8 * g8, N, act);
#pragma unroll
                    for (int i = 0; i < 8; ++i) v1[8 * g8 + i] = __float_as_uint(f[i]);
                }
            }
            uint32_t p[32];
#pragma unroll
            for (int i = 0; i < 16; ++i) p[i] = pack2<kBf16>(v0[2 * i], v0[2 * i + 1]);
#pragma unroll
            for (int i = 0; i < 16; ++i) p[16 + i] = pack2<kBf16>(v1[2 * i], v1[2 * i + 1]);
            store_chunk(p, m0, col0);
        };

        uint32_t acc = 0;
        bool ok = true;
        for (uint32_t item = 0; item < n_items; ++item, ++acc) {
            const WorkItem wi = work_item(split, cid, item);
            const TileCoord tc = tile_coord(wi.tile, num_m_blocks, num_n_blocks, group_m);
            const int32_t m0 = static_cast<int32_t>(tc.m_blk * C::MMA_M + rank * kBlockM);
            // a half-width item holds BN / 2 columns, from half a tile in for the second half
            const int32_t n0 = static_cast<int32_t>(
                tc.n_blk * C::BN +
                ((kHalves && wi.half != 0u) ? (wi.half - 1u) * (C::BN / 2u) : 0u));
            const bool rows_in = m0 < static_cast<int32_t>(M);
            const uint32_t b = acc % C::ACC_BUFS;
            const uint32_t aph = (acc / C::ACC_BUFS) & 1u;
            // One thread polls; the barrier-AND gives all 128 threads the same answer, so the
            // group never splits between leaving and waiting at a named barrier.
            uint32_t waited = 1u;
            if (et == 0) waited = mbar_wait<kPair>(tfull_bar(b), aph, abort_flag, timeout_ns);
            waited = named_barrier_and(2, C::EPI_THREADS, waited);
            if (!waited) {
                if (et == 0) report(kStatusEpilogueTimeout, abort_flag);
                ok = false;
                break;
            }
            tcgen05_fence_after();
            if constexpr (C::ACC_BUFS == 1) {
                if (!wi.partial) {
                    // One accumulator: read all of it out (as packed 16-bit values, after the
                    // fused epilogue), hand it back to the MMA issuer, then store.
                    uint32_t pk[C::BN / C::D_COLS][32];
#pragma unroll
                    for (uint32_t c = 0; c < C::BN / C::D_COLS; ++c) {
                        uint32_t v0[32], v1[32];
                        const uint32_t taddr = tmem_base + lane_off + c * C::D_COLS;
                        tmem_ld_32x32b_x32(taddr, v0, 0);
                        tmem_ld_32x32b_x32(taddr, v1, 32);
                        tmem_ld_wait();
                        const int32_t col0 = n0 + static_cast<int32_t>(c * C::D_COLS);
                        if (fused) {
#pragma unroll
                            for (int g8 = 0; g8 < 8; ++g8) {
                                float f[8];
#pragma unroll
                                for (int i = 0; i < 8; ++i)
                                    f[i] = __uint_as_float(g8 < 4 ? v0[8 * g8 + i]
                                                                  : v1[8 * (g8 - 4) + i]);
                                epilogue8<kBf16, false>(f, bias, col0 + 8 * g8, N, act);
#pragma unroll
                                for (int i = 0; i < 8; ++i) {
                                    if (g8 < 4) v0[8 * g8 + i] = __float_as_uint(f[i]);
                                    else v1[8 * (g8 - 4) + i] = __float_as_uint(f[i]);
                                }
                            }
                        }
#pragma unroll
                        for (int i = 0; i < 16; ++i) pk[c][i] = pack2<kBf16>(v0[2 * i], v0[2 * i + 1]);
#pragma unroll
                        for (int i = 0; i < 16; ++i)
                            pk[c][16 + i] = pack2<kBf16>(v1[2 * i], v1[2 * i + 1]);
                    }
                    tcgen05_fence_before();
                    __syncwarp();
                    if (lane == 0) {
                        if constexpr (kPair) mbar_arrive_remote(mapa_shared(tempty_bar(0), 0));
                        else mbar_arrive_local(tempty_bar(0));
                    }
                    __syncwarp();
#pragma unroll
                    for (uint32_t c = 0; c < C::BN / C::D_COLS; ++c) {
                        const int32_t col0 = n0 + static_cast<int32_t>(c * C::D_COLS);
                        if (col0 < static_cast<int32_t>(N) && rows_in) store_chunk(pk[c], m0, col0);
                    }
                    continue;
                }
            }
            if (!wi.partial) {
                // A whole tile: two 64-column chunks per round, both chunks' loads in flight
                // before one wait.
                constexpr uint32_t NC = C::BN / C::D_COLS;
                // chunks whose loads are in flight together: two for the wide tiles, one for
                // 128 columns (whose registers would not hold two with the rest of the kernel)
                constexpr uint32_t kBatch = NC >= 4 ? 2u : 1u;
                const uint32_t nc = (kHalves && wi.half != 0u) ? NC / 2u : NC;   // this item's chunks
#pragma unroll
                for (uint32_t c2 = 0; c2 < NC; c2 += kBatch) {
                    if (c2 >= nc) break;
                    uint32_t v[2 * kBatch][32];
                    const uint32_t taddr = tmem_base + lane_off + b * C::BN + c2 * C::D_COLS;
#pragma unroll
                    for (uint32_t h = 0; h < 2 * kBatch; ++h)
                        if (c2 + h / 2 < nc)
                            tmem_ld_32x32b_x32(taddr, v[h], static_cast<int>(32u * h));
                    tmem_ld_wait();
                    if (c2 + kBatch >= nc) hand_back(b);   // this warp is done with accumulator b
#pragma unroll
                    for (uint32_t cc = 0; cc < kBatch; ++cc) {
                        const uint32_t c = c2 + cc;
                        const int32_t col0 = n0 + static_cast<int32_t>(c * C::D_COLS);
                        if (c < nc && col0 < static_cast<int32_t>(N) && rows_in)
                            emit64(v[2 * cc], v[2 * cc + 1], m0, col0);
                    }
                }
                continue;
            }
            // Stream-K piece of tail tile r, whose k-blocks units u0 .. u1 share in order.  The
            // piece that starts the tile (k-block 0) finishes it: it adds the other pieces'
            // fp32 partial sums, in unit order, to its own and stores the tile.  That piece is
            // always its unit's last item, and every other piece of the tile is its unit's
            // first (or only) stream-K piece, which parks its partial sums in the unit's one
            // slot and raises its flag: so a finishing piece waits only for pieces that wait for
            // nothing (a unit's data-parallel tiles, before its pieces, wait for nothing either).
            const uint32_t r = wi.tile - (num_tiles - sk_tiles);
            const uint32_t u0 = sk_unit_of(split, r * num_k_blocks);
            const uint32_t u1 = sk_unit_of(split, r * num_k_blocks + num_k_blocks - 1u);
            const auto flag_of = [&](uint32_t u) {
                return sk_flags + (r * kMaxContrib + (u - u0)) * kCtaGroup + rank;
            };
            if (wi.kb0 != 0u) {
                float4* my_part = part_of(cid);
#pragma unroll 1
                for (uint32_t c = 0; c < C::BN / C::D_COLS; ++c) {
                    uint32_t v0[32], v1[32];
                    const uint32_t taddr = tmem_base + lane_off + b * C::BN + c * C::D_COLS;
                    tmem_ld_32x32b_x32(taddr, v0, 0);
                    tmem_ld_32x32b_x32(taddr, v1, 32);
                    tmem_ld_wait();
                    if (c == C::BN / C::D_COLS - 1) hand_back(b);
                    float4* dst = my_part + c * 16u * 128u + row;
#pragma unroll
                    for (uint32_t j = 0; j < 8; ++j)
                        dst[j * 128u] = make_float4(
                            __uint_as_float(v0[4 * j]), __uint_as_float(v0[4 * j + 1]),
                            __uint_as_float(v0[4 * j + 2]), __uint_as_float(v0[4 * j + 3]));
#pragma unroll
                    for (uint32_t j = 0; j < 8; ++j)
                        dst[(8 + j) * 128u] = make_float4(
                            __uint_as_float(v1[4 * j]), __uint_as_float(v1[4 * j + 1]),
                            __uint_as_float(v1[4 * j + 2]), __uint_as_float(v1[4 * j + 3]));
                }
                __threadfence();
                named_barrier_sync(1, C::EPI_THREADS);
                if (et == 0) {
                    __threadfence();
                    st_release_gpu(flag_of(cid), 1u);
                }
                continue;
            }
            // The finishing piece: every other contributor's partial sums must be in place.
            uint32_t ready = 1u;
            if (et == 0) {
                for (uint32_t u = u0 + 1u; u <= u1 && ready; ++u)
                    ready = wait_flag(flag_of(u), abort_flag, timeout_ns) ? 1u : 0u;
            }
            ready = named_barrier_and(2, C::EPI_THREADS, ready);
            if (!ready) {
                if (et == 0) report(kStatusEpilogueTimeout, abort_flag);
                ok = false;
                break;
            }
            __threadfence();
            // Up to kMaxContrib - 1 other pieces (the host bounds it); a slice's loads from all
            // of them are issued before any is added.
            const uint32_t nother = u1 - u0;
            const float4* srcs[kMaxContrib - 1];
#pragma unroll
            for (uint32_t q = 0; q < kMaxContrib - 1; ++q)
                srcs[q] = part_of(u0 + 1u + q <= u1 ? u0 + 1u + q : u1) + row;
#pragma unroll 1
            for (uint32_t c = 0; c < C::BN / C::D_COLS; ++c) {
                uint32_t v[2][32];
                const uint32_t taddr = tmem_base + lane_off + b * C::BN + c * C::D_COLS;
                tmem_ld_32x32b_x32(taddr, v[0], 0);
                tmem_ld_32x32b_x32(taddr, v[1], 32);
                tmem_ld_wait();
                if (c == C::BN / C::D_COLS - 1) hand_back(b);
#pragma unroll
                for (uint32_t h = 0; h < 4; ++h) {   // 16 columns (4 groups of 4) per step
                    float4 x[kMaxContrib - 1][4];
#pragma unroll
                    for (uint32_t q = 0; q < kMaxContrib - 1; ++q)
#pragma unroll
                        for (uint32_t j = 0; j < 4; ++j)
                            x[q][j] = q < nother
                                          ? __ldcg(srcs[q] + (c * 16u + h * 4u + j) * 128u)
                                          : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
                    for (uint32_t j = 0; j < 4; ++j) {
                        const uint32_t g = h * 4u + j;              // 16-byte group 0 .. 15
                        uint32_t* e = &v[g / 8u][(g % 8u) * 4u];    // its 4 fp32 values
                        float t0 = __uint_as_float(e[0]), t1 = __uint_as_float(e[1]);
                        float t2 = __uint_as_float(e[2]), t3 = __uint_as_float(e[3]);
#pragma unroll
                        for (uint32_t q = 0; q < kMaxContrib - 1; ++q) {
                            t0 += x[q][j].x;
                            t1 += x[q][j].y;
                            t2 += x[q][j].z;
                            t3 += x[q][j].w;
                        }
                        e[0] = __float_as_uint(t0);
                        e[1] = __float_as_uint(t1);
                        e[2] = __float_as_uint(t2);
                        e[3] = __float_as_uint(t3);
                    }
                }
                const int32_t col0 = n0 + static_cast<int32_t>(c * C::D_COLS);
                if (col0 < static_cast<int32_t>(N) && rows_in) emit64(v[0], v[1], m0, col0);
            }
        }
        (void)ok;
        if constexpr (kTmaStore) {
            // The staging buffers must outlive the copies that read them; the stores' writes
            // complete on their own before the grid does.
            if (et == 0) bulk_wait_group_read<0>();
        }
        __syncwarp();
    }

    // ---- teardown ------------------------------------------------------------------------
    // Every role of this CTA is done with tensor memory and with the shared memory that copies
    // and MMAs use.  In a pair, every operation one CTA aims at the other has been waited for
    // by its target by now (loads and MMA commits by the roles that consume them, the
    // epilogues' hand-backs by the MMA issuer above); the two TMEM owners still meet before
    // freeing their columns, through one barrier of each CTA (a cheaper rendezvous than the
    // cluster barrier, and a bounded one: its limit is a multiple of every role's own, so that
    // after a fault both CTAs still get here before it runs out).
    tcgen05_fence_before();
    __syncthreads();
    if (sk_tiles != 0u && threadIdx.x == 0) {
        // The last CTA of the launch to finish hands the other flag region to the next launch.
        __threadfence();
        if (atomicAdd(ws_hdr + 1, 1u) == gridDim.x - 1u) {
            atomicExch(ws_hdr + 1, 0u);
            atomicXor(ws_hdr, 1u);
        }
    }
    if (warp == 1) {
        if constexpr (kPair) {
            if (elect_one_sync()) {
                bool w;
                if (rank == 0) {
                    w = mbar_wait<kPair>(pair_bar, 0, nullptr, 4 * timeout_ns);
                    mbar_arrive_remote(mapa_shared(pair_bar, 1));
                } else {
                    mbar_arrive_remote(mapa_shared(pair_bar, 0));
                    w = mbar_wait<kPair>(pair_bar, 0, nullptr, 4 * timeout_ns);
                }
                if (!w) atomicOr(&gemm_f16_status_word, kStatusDrainTimeout);
            }
            __syncwarp();
        }
        tcgen05_fence_after();
        tmem_dealloc<kCtaGroup>(tmem_base, C::TMEM_COLS);
    }
}


// ==============================================================================================
// Block scales, row-major (rows x k_blocks bytes, one E8M0 code per row and 32-element K block)
// -> the tiled layout the block-scaled kernels read (mx_sf_offset).  One thread per byte of the
// tiled buffer; bytes that no (row, block) maps to (rows past the last 128-row group, K blocks
// past the last group of 4) get 127, a scale of 1.0, so a zero-filled K tail stays zero.
// ==============================================================================================
__global__ void mx_pack_scales_kernel(const uint8_t* __restrict__ src, uint8_t* __restrict__ dst,
                                      uint64_t rows, uint32_t k_blocks, uint32_t k_groups,
                                      uint64_t total)
{
    const uint64_t stride = static_cast<uint64_t>(gridDim.x) * blockDim.x;
    for (uint64_t t = static_cast<uint64_t>(blockIdx.x) * blockDim.x + threadIdx.x; t < total;
         t += stride) {
        const uint64_t chunk = t / 512u;
        const uint32_t w = static_cast<uint32_t>(t % 512u);
        const uint64_t row = (chunk / k_groups) * 128u + ((w % 16u) / 4u) * 32u + w / 16u;
        const uint32_t kb = static_cast<uint32_t>(chunk % k_groups) * 4u + w % 4u;
        dst[t] = (row < rows && kb < k_blocks) ? src[row * k_blocks + kb] : uint8_t{127};
    }
}

}  // namespace gf16
