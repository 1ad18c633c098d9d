// Gated Delta Net prefill on sm_103a (C ABI in include/gdn.h).
//
// The recurrence (page "TIRx" (zixuwang.me), section "用状态递推解释 GDN"), per sequence and
// value head, state H of shape [dv, dk]:
//     H_decay = alpha_t H;  prediction = H_decay k_t;  u_t = beta_t (v_t - prediction);
//     H = H_decay + u_t k_t^T;  o_t = scale H q_t.
// The page's GPU form works on 64-token chunks: matrix products build the chunk's QK, KK and WY
// data, then a state scan produces the outputs.  This file follows that plan:
//
// Within a chunk with cumulative decays g_t = alpha_1 ... alpha_t and start state H0,
//     H_t = g_t H0 + sum_{s<=t} (g_t / g_s) u_s k_s^T,
// so the updates u_t satisfy (I + L) U = diag(beta) V - diag(beta g) K H0^T with the strictly
// lower triangular L[t][s] = beta_t (g_t / g_s) (k_t . k_s).  With T = (I + L)^-1,
//     W = T diag(beta g) K      (C x dk)      U' = T diag(beta) V      (C x dv)
// depend on the chunk alone (gdn_prepare_kernel, all chunks in parallel), and the scan over a
// sequence's chunks (gdn_scan_kernel) computes
//     U = U' - W H0^T,   O = scale (diag(g) Q H0^T + A U),   H_next = g_C H0 + U^T diag(g_C / g) K
// with A[t][s] = (g_t / g_s) (q_t . k_s) for s <= t.  Every value row of H evolves on its own,
// so the scan splits a head's dv rows over several CTAs.
//
// A sequence's last chunk may be short: its missing tokens are read as q = k = v = 0,
// alpha = 1, beta = 0 (the page's rule for packed tails), which leaves the state and the valid
// outputs unchanged.  All arithmetic is fp32; q, k, v and o are bfloat16.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdarg>
#include <cstdint>
#include <cstdio>
#include <string>

#include "../../include/gdn.h"

namespace {

constexpr int kC = 64;          // tokens per chunk
constexpr int kD = 128;         // head dimension (dk = dv)
constexpr int kRows = 16;       // value rows of the state per scan CTA

thread_local std::string t_gdn_error;

int gdn_fail(int code, const char* fmt, ...)
{
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    std::vsnprintf(buf, sizeof(buf), fmt, ap);
    va_end(ap);
    t_gdn_error = buf;
    return code;
}

int64_t max_chunks_for(int64_t T, int64_t n) { return T / kC + n; }

// Workspace layout (all offsets 256-byte aligned).
struct WsLayout {
    size_t chunk_offset, n_chunks, chunks, wt, ut, at, gam, total;
};

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

WsLayout layout_for(int64_t T, int64_t n, int64_t h_v)
{
    const size_t mc = static_cast<size_t>(max_chunks_for(T, n));
    WsLayout l{};
    size_t o = 0;
    l.chunk_offset = o; o = align256(o + sizeof(int32_t) * static_cast<size_t>(n + 1));
    l.n_chunks = o;     o = align256(o + sizeof(int32_t));
    l.chunks = o;       o = align256(o + sizeof(int4) * mc);
    l.wt = o;           o = align256(o + sizeof(float) * mc * h_v * kD * kC);
    l.ut = o;           o = align256(o + sizeof(float) * mc * h_v * kD * kC);
    l.at = o;           o = align256(o + sizeof(float) * mc * h_v * kC * kC);
    l.gam = o;          o = align256(o + sizeof(float) * mc * h_v * kC);
    l.total = o;
    return l;
}

// ---- chunk list: per sequence, ceil(len / 64) chunks, numbered in sequence order -------------
__global__ void gdn_chunk_list_kernel(const int32_t* __restrict__ cu, int32_t n_seqs,
                                      int32_t* __restrict__ chunk_offset, int4* __restrict__ chunks,
                                      int32_t max_chunks, int32_t* __restrict__ n_chunks)
{
    __shared__ int32_t scan[1024];
    __shared__ int32_t carry;
    if (threadIdx.x == 0) carry = 0;
    __syncthreads();
    for (int32_t base = 0; base < n_seqs; base += blockDim.x) {
        const int32_t i = base + static_cast<int32_t>(threadIdx.x);
        int32_t nc = 0, start = 0, len = 0;
        if (i < n_seqs) {
            start = cu[i];
            len = cu[i + 1] - start;
            nc = len > 0 ? (len + kC - 1) / kC : 0;
        }
        scan[threadIdx.x] = nc;
        __syncthreads();
        for (int32_t d = 1; d < static_cast<int32_t>(blockDim.x); d <<= 1) {   // inclusive scan
            const int32_t add = threadIdx.x >= static_cast<uint32_t>(d) ? scan[threadIdx.x - d] : 0;
            __syncthreads();
            scan[threadIdx.x] += add;
            __syncthreads();
        }
        const int32_t first = carry + scan[threadIdx.x] - nc;
        if (i < n_seqs) {
            chunk_offset[i] = first;
            for (int32_t c = 0; c < nc && first + c < max_chunks; ++c) {
                const int32_t l = len - c * kC < kC ? len - c * kC : kC;
                chunks[first + c] = make_int4(i, start + c * kC, l, 0);
            }
        }
        __syncthreads();
        if (threadIdx.x == blockDim.x - 1) carry += scan[threadIdx.x];
        __syncthreads();
    }
    if (threadIdx.x == 0) {
        chunk_offset[n_seqs] = carry;
        *n_chunks = carry;
    }
}

__device__ __forceinline__ float bf16_at(const __nv_bfloat16* p)
{
    return __uint_as_float(static_cast<uint32_t>(*reinterpret_cast<const uint16_t*>(p)) << 16);
}

// 16-byte global -> shared copy that completes asynchronously; src_bytes = 0 writes zeros.
__device__ __forceinline__ void cp_async16(void* smem_dst, const void* gmem_src, uint32_t src_bytes)
{
    const uint32_t d = static_cast<uint32_t>(__cvta_generic_to_shared(smem_dst));
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(d), "l"(gmem_src),
                 "r"(src_bytes)
                 : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_group 0;" ::: "memory"); }

// d += a * b for a 16 x 16 (k) bf16 A fragment and a 16 (k) x 8 bf16 B fragment (m16n8k16,
// fp32 accumulation); each 32-bit register holds two consecutive-k elements.
__device__ __forceinline__ void mma_bf16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1)
{
    asm volatile("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, "
                 "{%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
                 : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
                 : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Rows of 128 bf16 in shared memory are padded to 136 elements (272 bytes): rows 16 apart then
// start 4 banks apart, so the strided tiles below read them without bank conflicts.
constexpr int kRowB = 136;

// ---- per (chunk, value head): W^T, U'^T, A^T and the cumulative decays ----------------------
// K, Q, V of the chunk sit in shared memory as padded bf16 rows.  Products K K^T and Q K^T run
// on the tensor cores (bf16 operands, exact products).  Then (I + L) X = R
// is solved for the 256 right-hand-side columns R = [diag(beta g) K | diag(beta) V] by forward
// substitution, one column per thread with the column held in registers: no inverse is formed
// and no barrier is needed inside the solve.
constexpr int kPrepThreads = 256;
constexpr size_t kPrepSmem =
    sizeof(__nv_bfloat16) * 3 * kC * kRowB + sizeof(float) * (kC * kC + kC * (kC + 1) + 4 * kC);

__global__ void __launch_bounds__(kPrepThreads, 2)
    gdn_prepare_kernel(const __nv_bfloat16* __restrict__ q, const __nv_bfloat16* __restrict__ k,
                       const __nv_bfloat16* __restrict__ v, const float* __restrict__ alpha,
                       const float* __restrict__ beta, const int4* __restrict__ chunks,
                       const int32_t* __restrict__ n_chunks, int32_t h_qk, int32_t h_v,
                       float* __restrict__ wt, float* __restrict__ ut, float* __restrict__ at,
                       float* __restrict__ gam_out)
{
    const int32_t ch = blockIdx.x;
    const int32_t j = blockIdx.y;
    if (ch >= *n_chunks) return;
    const int4 info = chunks[ch];
    const int32_t t0 = info.y, len = info.z;
    const int32_t jq = j / (h_v / h_qk);
    extern __shared__ __align__(16) uint8_t smraw[];
    __nv_bfloat16* Kb = reinterpret_cast<__nv_bfloat16*>(smraw);   // [64][136]
    __nv_bfloat16* Qb = Kb + kC * kRowB;
    __nv_bfloat16* Vb = Qb + kC * kRowB;
    float* Ls = reinterpret_cast<float*>(Vb + kC * kRowB);          // [64][64] L, strictly lower
    float* As = Ls + kC * kC;                                         // [64 s][65] A transposed
    float* g = As + kC * (kC + 1);
    float* bt = g + kC;
    float* bg = bt + kC;
    float* al = bg + kC;
    const int tid = threadIdx.x;

    for (int idx = tid; idx < kC * 16; idx += kPrepThreads) {
        const int t = idx / 16, p = idx % 16;
        const bool valid = t < len;
        const int64_t tok = static_cast<int64_t>(t0) + (valid ? t : 0);
        const uint32_t nb = valid ? 16u : 0u;
        cp_async16(Kb + t * kRowB + p * 8, k + (tok * h_qk + jq) * kD + p * 8, nb);
        cp_async16(Qb + t * kRowB + p * 8, q + (tok * h_qk + jq) * kD + p * 8, nb);
        cp_async16(Vb + t * kRowB + p * 8, v + (tok * h_v + j) * kD + p * 8, nb);
    }
    cp_async_commit();
    if (tid < kC) {
        const bool valid = tid < len;
        const int64_t tok = static_cast<int64_t>(t0) + tid;
        al[tid] = valid ? alpha[tok * h_v + j] : 1.f;
        bt[tid] = valid ? beta[tok * h_v + j] : 0.f;
    }
    __syncthreads();
    if (tid < 32) {
        // running products of alpha: each lane multiplies two, then a warp product scan
        float a0 = al[2 * tid], a1 = al[2 * tid + 1];
        float p = a0 * a1;
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
            const float o = __shfl_up_sync(0xffffffffu, p, d);
            if (tid >= d) p *= o;
        }
        float before = __shfl_up_sync(0xffffffffu, p, 1);
        if (tid == 0) before = 1.f;
        g[2 * tid] = before * a0;
        g[2 * tid + 1] = p;
    }
    cp_async_wait_all();
    __syncthreads();
    if (tid < kC) bg[tid] = bt[tid] * g[tid];

    // K K^T and Q K^T on the tensor cores: mma.sync m16n8k16 with bf16 operands (exact products,
    // fp32 sums).  Warp w owns rows 16 (w / 2) .. + 15 and columns 32 (w % 2) .. + 31 of both.
    {
        const int warp = tid / 32, lane = tid % 32;
        const int gq = lane >> 2, tg = lane & 3;
        const int m0 = 16 * (warp >> 1), nb = 32 * (warp & 1);
        float kk[4][4] = {}, qk[4][4] = {};
        const auto ld32 = [](const __nv_bfloat16* p) { return *reinterpret_cast<const uint32_t*>(p); };
#pragma unroll
        for (int k0 = 0; k0 < kD; k0 += 16) {
            const uint32_t ka0 = ld32(Kb + (m0 + gq) * kRowB + k0 + 2 * tg);
            const uint32_t ka1 = ld32(Kb + (m0 + gq + 8) * kRowB + k0 + 2 * tg);
            const uint32_t ka2 = ld32(Kb + (m0 + gq) * kRowB + k0 + 2 * tg + 8);
            const uint32_t ka3 = ld32(Kb + (m0 + gq + 8) * kRowB + k0 + 2 * tg + 8);
            const uint32_t qa0 = ld32(Qb + (m0 + gq) * kRowB + k0 + 2 * tg);
            const uint32_t qa1 = ld32(Qb + (m0 + gq + 8) * kRowB + k0 + 2 * tg);
            const uint32_t qa2 = ld32(Qb + (m0 + gq) * kRowB + k0 + 2 * tg + 8);
            const uint32_t qa3 = ld32(Qb + (m0 + gq + 8) * kRowB + k0 + 2 * tg + 8);
#pragma unroll
            for (int nt = 0; nt < 4; ++nt) {
                const int n0 = nb + 8 * nt;
                const uint32_t b0 = ld32(Kb + (n0 + gq) * kRowB + k0 + 2 * tg);
                const uint32_t b1 = ld32(Kb + (n0 + gq) * kRowB + k0 + 2 * tg + 8);
                mma_bf16(kk[nt], ka0, ka1, ka2, ka3, b0, b1);
                mma_bf16(qk[nt], qa0, qa1, qa2, qa3, b0, b1);
            }
        }
#pragma unroll
        for (int nt = 0; nt < 4; ++nt) {
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int t = m0 + gq + 8 * (e >> 1);
                const int s = nb + 8 * nt + 2 * tg + (e & 1);
                const float ratio = s <= t ? g[t] / g[s] : 0.f;
                Ls[t * kC + s] = s < t ? bt[t] * ratio * kk[nt][e] : 0.f;
                As[s * (kC + 1) + t] = ratio * qk[nt][e];
            }
        }
    }
    __syncthreads();

    // A^T to global, coalesced
    {
        float* atc = at + (static_cast<int64_t>(ch) * h_v + j) * kC * kC;
        for (int e = tid; e < kC * kC; e += kPrepThreads)
            atc[e] = As[(e / kC) * (kC + 1) + e % kC];
    }

    // (I + L) X = R by forward substitution, one right-hand-side column per thread
    {
        const bool isw = tid < kD;
        const int col = tid & (kD - 1);
        const __nv_bfloat16* src = isw ? Kb : Vb;
        const float* sc = isw ? bg : bt;
        float x[kC];
#pragma unroll
        for (int t = 0; t < kC; ++t) {
            float acc[4] = {sc[t] * bf16_at(src + t * kRowB + col), 0.f, 0.f, 0.f};
#pragma unroll
            for (int s4 = 0; s4 < (t & ~3); s4 += 4) {
                const float4 l = *reinterpret_cast<const float4*>(Ls + t * kC + s4);
                acc[0] = fmaf(-l.x, x[s4], acc[0]);
                acc[1] = fmaf(-l.y, x[s4 + 1], acc[1]);
                acc[2] = fmaf(-l.z, x[s4 + 2], acc[2]);
                acc[3] = fmaf(-l.w, x[s4 + 3], acc[3]);
            }
#pragma unroll
            for (int s = t & ~3; s < t; ++s) acc[0] = fmaf(-Ls[t * kC + s], x[s], acc[0]);
            x[t] = (acc[0] + acc[1]) + (acc[2] + acc[3]);
        }
        float* dst = (isw ? wt : ut) + ((static_cast<int64_t>(ch) * h_v + j) * kD + col) * kC;
#pragma unroll
        for (int t = 0; t < kC; t += 4)
            *reinterpret_cast<float4*>(dst + t) = make_float4(x[t], x[t + 1], x[t + 2], x[t + 3]);
    }
    if (tid < kC) gam_out[(static_cast<int64_t>(ch) * h_v + j) * kC + tid] = g[tid];
}

// ---- per (sequence, value head, block of 16 value rows): the state scan over the chunks -----
// The chunk's inputs are double-buffered: while chunk c is computed, cp.async brings chunk
// c + 1 (W^T, A^T, the block's U'^T rows, decays, and q/k as padded bf16 rows).  The three
// products run on the tensor cores (mma.sync m16n8k8, TF32 inputs, fp32 accumulation), each
// warp owning 16 x 8 output tiles.  Operands that are fp32 (W, A, the state, U, the decayed
// keys) are split into a TF32 high part and the TF32 rounding of the rest, and each product
// takes three passes (hi*hi + hi*lo + lo*hi), which keeps fp32 accuracy; q and k are bfloat16,
// exact in TF32, so their passes need no split.
constexpr int kScanThreads = 256;
constexpr int kRowW = 72;          // padded W^T / A^T rows (floats): fragment loads hit 32 banks
constexpr int kRowS = 24;          // padded S^T / U^T rows (floats)
struct ScanBuf {
    float wt[kD * kRowW];          // W^T [c][t]
    float at[kC * kRowW];          // A^T [s][t]
    float up[kRows * kC];          // U'^T rows r0 .. r0+15, [r][t]
    float g[kC];
    __nv_bfloat16 qb[kC * kRowB];  // q rows, padded
    __nv_bfloat16 kb[kC * kRowB];  // k rows, padded
};
constexpr size_t kScanSmem = 2 * sizeof(ScanBuf) + sizeof(float) * (kD * kRowS + kC * kRowS + kC);

__device__ __forceinline__ void scan_prefetch(ScanBuf& b, const __nv_bfloat16* __restrict__ q,
                                              const __nv_bfloat16* __restrict__ k,
                                              const float* __restrict__ wt,
                                              const float* __restrict__ ut,
                                              const float* __restrict__ at,
                                              const float* __restrict__ gam, int64_t cj,
                                              int32_t r0, int32_t t0, int32_t len, int32_t h_qk,
                                              int32_t jq, int tid)
{
    const float* w = wt + cj * kD * kC;
    for (int e = tid; e < kD * kC / 4; e += kScanThreads)
        cp_async16(b.wt + (e / 16) * kRowW + (e % 16) * 4, w + 4 * e, 16);
    const float* a = at + cj * kC * kC;
    for (int e = tid; e < kC * kC / 4; e += kScanThreads)
        cp_async16(b.at + (e / 16) * kRowW + (e % 16) * 4, a + 4 * e, 16);
    const float* u = ut + (cj * kD + r0) * kC;
    for (int e = tid; e < kRows * kC / 4; e += kScanThreads) cp_async16(b.up + 4 * e, u + 4 * e, 16);
    if (tid < kC / 4) cp_async16(b.g + 4 * tid, gam + cj * kC + 4 * tid, 16);
    for (int idx = tid; idx < kC * 16; idx += kScanThreads) {
        const int t = idx / 16, p = idx % 16;
        const bool valid = t < len;
        const int64_t tok = static_cast<int64_t>(t0) + (valid ? t : 0);
        cp_async16(b.qb + t * kRowB + p * 8, q + (tok * h_qk + jq) * kD + p * 8, valid ? 16u : 0u);
        cp_async16(b.kb + t * kRowB + p * 8, k + (tok * h_qk + jq) * kD + p * 8, valid ? 16u : 0u);
    }
    cp_async_commit();
}

__device__ __forceinline__ uint32_t tf32_rna(float x)
{
    uint32_t r;
    asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(x));
    return r;
}

// x = hi + lo with hi, lo TF32 values (lo the TF32 rounding of x - hi)
__device__ __forceinline__ void split_tf32(float x, uint32_t& hi, uint32_t& lo)
{
    hi = tf32_rna(x);
    lo = tf32_rna(x - __uint_as_float(hi));
}

// d += a * b for a 16 x 8 (k) A fragment and an 8 (k) x 8 B fragment (m16n8k8, TF32 -> f32)
__device__ __forceinline__ void mma_tf32(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1)
{
    asm volatile("mma.sync.aligned.m16n8k8.row.col.f32.tf32.tf32.f32 {%0, %1, %2, %3}, "
                 "{%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
                 : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
                 : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// d += A * B with fp32 A (a[4]) and B (b[2]) fragments, three TF32 passes
__device__ __forceinline__ void mma_3xtf32(float (&d)[4], const float (&a)[4], const float (&b)[2])
{
    uint32_t ah[4], al[4], bh[2], bl[2];
#pragma unroll
    for (int i = 0; i < 4; ++i) split_tf32(a[i], ah[i], al[i]);
#pragma unroll
    for (int i = 0; i < 2; ++i) split_tf32(b[i], bh[i], bl[i]);
    mma_tf32(d, al[0], al[1], al[2], al[3], bh[0], bh[1]);
    mma_tf32(d, ah[0], ah[1], ah[2], ah[3], bl[0], bl[1]);
    mma_tf32(d, ah[0], ah[1], ah[2], ah[3], bh[0], bh[1]);
}

__global__ void __launch_bounds__(kScanThreads, 1)
    gdn_scan_kernel(const __nv_bfloat16* __restrict__ q, const __nv_bfloat16* __restrict__ k,
                    const int32_t* __restrict__ cu, const int32_t* __restrict__ chunk_offset,
                    const float* __restrict__ wt, const float* __restrict__ ut,
                    const float* __restrict__ at, const float* __restrict__ gam,
                    const float* __restrict__ s0, float* __restrict__ s_final,
                    __nv_bfloat16* __restrict__ o, int32_t h_qk, int32_t h_v, float scale)
{
    const int32_t i = blockIdx.x;
    const int32_t j = blockIdx.y;
    const int32_t r0 = blockIdx.z * kRows;
    const int32_t jq = j / (h_v / h_qk);
    extern __shared__ __align__(16) uint8_t smraw[];
    ScanBuf* buf = reinterpret_cast<ScanBuf*>(smraw);
    float* St = reinterpret_cast<float*>(buf + 2);  // state transposed [c][r], 128 x 16 (+pad)
    float* Ut = St + kD * kRowS;                    // U transposed [s][r], 64 x 16 (+pad)
    float* kf = Ut + kC * kRowS;                    // [64] g_C / g_s
    const int tid = threadIdx.x;
    const int warp = tid / 32, lane = tid % 32;
    const int gq = lane >> 2, tg = lane & 3;        // fragment row group, thread in group

    const int64_t sbase = ((static_cast<int64_t>(i) * h_v + j) * kD + r0) * kD;
    for (int e = tid; e < kRows * kD; e += kScanThreads)
        St[(e % kD) * kRowS + e / kD] = s0 ? s0[sbase + e] : 0.f;

    const int32_t c_begin = chunk_offset[i], c_end = chunk_offset[i + 1];
    const int32_t seq_start = cu[i], seq_end = cu[i + 1];
    const auto chunk_t0 = [&](int32_t ch) { return seq_start + (ch - c_begin) * kC; };
    if (c_begin < c_end)
        scan_prefetch(buf[0], q, k, wt, ut, at, gam, static_cast<int64_t>(c_begin) * h_v + j, r0,
                      chunk_t0(c_begin), min(kC, seq_end - chunk_t0(c_begin)), h_qk, jq, tid);
    // U and O: warp tile rows (tokens) m0 .. m0+15, columns (state rows) n0 .. n0+7
    const int m0 = 16 * (warp >> 1), n0 = 8 * (warp & 1);
    for (int32_t ch = c_begin; ch < c_end; ++ch) {
        const int b = (ch - c_begin) & 1;
        const int32_t t0 = chunk_t0(ch);
        const int32_t len = min(kC, seq_end - t0);
        cp_async_wait_all();
        __syncthreads();   // chunk ch has landed; everyone is done with the other buffer
        if (ch + 1 < c_end)
            scan_prefetch(buf[b ^ 1], q, k, wt, ut, at, gam, static_cast<int64_t>(ch + 1) * h_v + j,
                          r0, chunk_t0(ch + 1), min(kC, seq_end - chunk_t0(ch + 1)), h_qk, jq, tid);
        const ScanBuf& B = buf[b];
        if (tid < kC) kf[tid] = B.g[kC - 1] / B.g[tid];

        // U = U' - W S^T  (M = tokens, N = state rows, K = c)
        {
            float d[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 4
            for (int k0 = 0; k0 < kD; k0 += 8) {
                const float a[4] = {B.wt[(k0 + tg) * kRowW + m0 + gq],
                                    B.wt[(k0 + tg) * kRowW + m0 + gq + 8],
                                    B.wt[(k0 + tg + 4) * kRowW + m0 + gq],
                                    B.wt[(k0 + tg + 4) * kRowW + m0 + gq + 8]};
                const float bb[2] = {St[(k0 + tg) * kRowS + n0 + gq],
                                     St[(k0 + tg + 4) * kRowS + n0 + gq]};
                mma_3xtf32(d, a, bb);
            }
            const int t = m0 + gq, r = n0 + 2 * tg;
            Ut[t * kRowS + r] = B.up[r * kC + t] - d[0];
            Ut[t * kRowS + r + 1] = B.up[(r + 1) * kC + t] - d[1];
            Ut[(t + 8) * kRowS + r] = B.up[r * kC + t + 8] - d[2];
            Ut[(t + 8) * kRowS + r + 1] = B.up[(r + 1) * kC + t + 8] - d[3];
        }
        __syncthreads();   // U complete

        // O = scale (diag(g) Q S^T + A U)
        {
            float qs[4] = {0.f, 0.f, 0.f, 0.f}, au[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 4
            for (int k0 = 0; k0 < kD; k0 += 8) {
                // q is bf16: exact in TF32, so only the state needs a split
                const uint32_t a0 = __float_as_uint(bf16_at(B.qb + (m0 + gq) * kRowB + k0 + tg));
                const uint32_t a1 = __float_as_uint(bf16_at(B.qb + (m0 + gq + 8) * kRowB + k0 + tg));
                const uint32_t a2 = __float_as_uint(bf16_at(B.qb + (m0 + gq) * kRowB + k0 + tg + 4));
                const uint32_t a3 =
                    __float_as_uint(bf16_at(B.qb + (m0 + gq + 8) * kRowB + k0 + tg + 4));
                uint32_t bh0, bl0, bh1, bl1;
                split_tf32(St[(k0 + tg) * kRowS + n0 + gq], bh0, bl0);
                split_tf32(St[(k0 + tg + 4) * kRowS + n0 + gq], bh1, bl1);
                mma_tf32(qs, a0, a1, a2, a3, bl0, bl1);
                mma_tf32(qs, a0, a1, a2, a3, bh0, bh1);
            }
            for (int k0 = 0; k0 < m0 + 16; k0 += 8) {   // A[t][s] = 0 for s > t
                const float a[4] = {B.at[(k0 + tg) * kRowW + m0 + gq],
                                    B.at[(k0 + tg) * kRowW + m0 + gq + 8],
                                    B.at[(k0 + tg + 4) * kRowW + m0 + gq],
                                    B.at[(k0 + tg + 4) * kRowW + m0 + gq + 8]};
                const float bb[2] = {Ut[(k0 + tg) * kRowS + n0 + gq],
                                     Ut[(k0 + tg + 4) * kRowS + n0 + gq]};
                mma_3xtf32(au, a, bb);
            }
            const int t = m0 + gq, r = n0 + 2 * tg;
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int tt = t + 8 * h;
                if (tt < len) {
                    const float gt = B.g[tt];
                    const __nv_bfloat162 v2 =
                        __floats2bfloat162_rn(scale * fmaf(gt, qs[2 * h], au[2 * h]),
                                              scale * fmaf(gt, qs[2 * h + 1], au[2 * h + 1]));
                    *reinterpret_cast<__nv_bfloat162*>(
                        o + ((static_cast<int64_t>(t0) + tt) * h_v + j) * kD + r0 + r) = v2;
                }
            }
        }
        __syncthreads();   // every reader of S is done before the update

        // S^T_next = g_C S^T + Kd^T U with Kd[s][c] = (g_C / g_s) K[s][c]  (M = c, N = rows, K = s)
        {
            const float gC = B.g[kC - 1];
            const int mc = 16 * warp;                 // state columns mc .. mc + 15
#pragma unroll
            for (int nt = 0; nt < 2; ++nt) {
                const int nn = 8 * nt;
                const int c = mc + gq, r = nn + 2 * tg;
                float d[4] = {gC * St[c * kRowS + r], gC * St[c * kRowS + r + 1],
                              gC * St[(c + 8) * kRowS + r], gC * St[(c + 8) * kRowS + r + 1]};
#pragma unroll 2
                for (int k0 = 0; k0 < kC; k0 += 8) {
                    const float f0 = kf[k0 + tg], f1 = kf[k0 + tg + 4];
                    const float a[4] = {f0 * bf16_at(B.kb + (k0 + tg) * kRowB + mc + gq),
                                        f0 * bf16_at(B.kb + (k0 + tg) * kRowB + mc + gq + 8),
                                        f1 * bf16_at(B.kb + (k0 + tg + 4) * kRowB + mc + gq),
                                        f1 * bf16_at(B.kb + (k0 + tg + 4) * kRowB + mc + gq + 8)};
                    const float bb[2] = {Ut[(k0 + tg) * kRowS + nn + gq],
                                         Ut[(k0 + tg + 4) * kRowS + nn + gq]};
                    mma_3xtf32(d, a, bb);
                }
                St[c * kRowS + r] = d[0];
                St[c * kRowS + r + 1] = d[1];
                St[(c + 8) * kRowS + r] = d[2];
                St[(c + 8) * kRowS + r + 1] = d[3];
            }
        }
    }
    cp_async_wait_all();
    __syncthreads();
    if (s_final)
        for (int e = tid; e < kRows * kD; e += kScanThreads)
            s_final[sbase + e] = St[(e % kD) * kRowS + e / kD];
}

bool misaligned(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) != 0; }

int check(const void* q, const void* k, const void* v, const float* alpha, const float* beta,
          const int32_t* cu, int64_t n_seqs, int64_t T, int64_t h_qk, int64_t h_v,
          int64_t head_dim, const void* o)
{
    if (n_seqs < 0 || T < 0 || h_qk <= 0 || h_v <= 0)
        return gdn_fail(GDN_ERR_INVALID_ARG, "negative size or no heads (n_seqs=%lld T=%lld "
                        "h_qk=%lld h_v=%lld)", (long long)n_seqs, (long long)T,
                        (long long)h_qk, (long long)h_v);
    if (h_v % h_qk != 0)
        return gdn_fail(GDN_ERR_INVALID_ARG, "h_v=%lld is not a multiple of h_qk=%lld",
                        (long long)h_v, (long long)h_qk);
    if (head_dim != kD)
        return gdn_fail(GDN_ERR_UNSUPPORTED, "head_dim=%lld; this build supports 128",
                        (long long)head_dim);
    if (T > (1ll << 30) || n_seqs > (1ll << 30) || h_v > 65535)
        return gdn_fail(GDN_ERR_INVALID_ARG, "size out of range");
    if (n_seqs == 0) return GDN_OK;
    if (cu == nullptr) return gdn_fail(GDN_ERR_INVALID_ARG, "cu_seqlens is null");
    if (T > 0 && (!q || !k || !v || !alpha || !beta || !o))
        return gdn_fail(GDN_ERR_INVALID_ARG, "a tensor pointer is null");
    if (T > 0 && (misaligned(q) || misaligned(k) || misaligned(v) || misaligned(o)))
        return gdn_fail(GDN_ERR_UNSUPPORTED, "q, k, v and o must be 16-byte aligned");
    return GDN_OK;
}

}  // namespace

extern "C" {

int gdn_prefill_workspace_bytes(int64_t total_tokens, int64_t n_seqs, int64_t h_v,
                                size_t* bytes)
{
    if (!bytes) return gdn_fail(GDN_ERR_INVALID_ARG, "bytes is null");
    if (total_tokens < 0 || n_seqs < 0 || h_v <= 0)
        return gdn_fail(GDN_ERR_INVALID_ARG, "negative size");
    *bytes = layout_for(total_tokens, n_seqs, h_v).total;
    return GDN_OK;
}

int gdn_prefill(const void* q, const void* k, const void* v, const float* alpha,
                const float* beta, const int32_t* cu_seqlens, int64_t n_seqs,
                int64_t total_tokens, int64_t h_qk, int64_t h_v, int64_t head_dim, float scale,
                const float* initial_state, void* o, float* final_state, void* workspace,
                size_t workspace_bytes, cudaStream_t stream)
{
    t_gdn_error.clear();
    int rc = check(q, k, v, alpha, beta, cu_seqlens, n_seqs, total_tokens, h_qk, h_v, head_dim,
                   o);
    if (rc != GDN_OK || n_seqs == 0) return rc;
    const WsLayout l = layout_for(total_tokens, n_seqs, h_v);
    if (workspace == nullptr || workspace_bytes < l.total || misaligned(workspace))
        return gdn_fail(GDN_ERR_INVALID_ARG, "workspace of %zu bytes (16-byte aligned) needed",
                        l.total);
    auto* ws = static_cast<uint8_t*>(workspace);
    auto* chunk_offset = reinterpret_cast<int32_t*>(ws + l.chunk_offset);
    auto* n_chunks = reinterpret_cast<int32_t*>(ws + l.n_chunks);
    auto* chunks = reinterpret_cast<int4*>(ws + l.chunks);
    auto* wt = reinterpret_cast<float*>(ws + l.wt);
    auto* ut = reinterpret_cast<float*>(ws + l.ut);
    auto* at = reinterpret_cast<float*>(ws + l.at);
    auto* gm = reinterpret_cast<float*>(ws + l.gam);
    const int64_t mc = max_chunks_for(total_tokens, n_seqs);

    static bool attrs = false;
    if (!attrs) {
        cudaFuncSetAttribute(gdn_prepare_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(kPrepSmem));
        cudaFuncSetAttribute(gdn_scan_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(kScanSmem));
        attrs = true;
    }
    gdn_chunk_list_kernel<<<1, 1024, 0, stream>>>(cu_seqlens, static_cast<int32_t>(n_seqs),
                                                  chunk_offset, chunks, static_cast<int32_t>(mc),
                                                  n_chunks);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess)
        return gdn_fail(GDN_ERR_CUDA, "gdn_chunk_list_kernel: %s", cudaGetErrorString(e));
    if (mc > 0 && total_tokens > 0) {
        const dim3 pgrid(static_cast<uint32_t>(mc), static_cast<uint32_t>(h_v));
        gdn_prepare_kernel<<<pgrid, kPrepThreads, kPrepSmem, stream>>>(
            static_cast<const __nv_bfloat16*>(q), static_cast<const __nv_bfloat16*>(k),
            static_cast<const __nv_bfloat16*>(v), alpha, beta, chunks, n_chunks,
            static_cast<int32_t>(h_qk), static_cast<int32_t>(h_v), wt, ut, at, gm);
        if ((e = cudaGetLastError()) != cudaSuccess)
            return gdn_fail(GDN_ERR_CUDA, "gdn_prepare_kernel: %s", cudaGetErrorString(e));
    }
    const dim3 sgrid(static_cast<uint32_t>(n_seqs), static_cast<uint32_t>(h_v), kD / kRows);
    gdn_scan_kernel<<<sgrid, kScanThreads, kScanSmem, stream>>>(
        static_cast<const __nv_bfloat16*>(q), static_cast<const __nv_bfloat16*>(k), cu_seqlens,
        chunk_offset, wt, ut, at, gm, initial_state, final_state,
        static_cast<__nv_bfloat16*>(o), static_cast<int32_t>(h_qk), static_cast<int32_t>(h_v),
        scale);
    if ((e = cudaGetLastError()) != cudaSuccess)
        return gdn_fail(GDN_ERR_CUDA, "gdn_scan_kernel: %s", cudaGetErrorString(e));
    return GDN_OK;
}

const char* gdn_last_error(void) { return t_gdn_error.c_str(); }

}  // extern "C"
