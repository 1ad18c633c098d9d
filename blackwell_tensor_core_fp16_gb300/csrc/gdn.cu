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
constexpr int kPad = kD + 1;    // padded row length of [64][128] tiles in shared memory

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

__device__ __forceinline__ void load_row_bf16(float* dst, const __nv_bfloat16* src, bool valid,
                                              int lane16)
{
    // 128 bf16 = 16 x 16 bytes; lane16 = 0..15 loads one 16-byte piece
    float f[8];
    if (valid) {
        const uint4 w = __ldg(reinterpret_cast<const uint4*>(src) + lane16);
        const uint32_t u[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            f[2 * i] = __uint_as_float(u[i] << 16);
            f[2 * i + 1] = __uint_as_float(u[i] & 0xFFFF0000u);
        }
    } else {
#pragma unroll
        for (int i = 0; i < 8; ++i) f[i] = 0.f;
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) dst[lane16 * 8 + i] = f[i];
}

// ---- per (chunk, value head): W^T, U'^T, A^T and the cumulative decays ----------------------
constexpr int kPrepThreads = 256;
constexpr size_t kPrepSmem = sizeof(float) * (3 * kC * kPad + 2 * kC * (kC + 1) + 3 * kC);

__global__ void __launch_bounds__(kPrepThreads, 1)
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
    extern __shared__ float sm[];
    float* Ks = sm;                       // [64][129]
    float* Qs = Ks + kC * kPad;           // [64][129]
    float* Vs = Qs + kC * kPad;           // [64][129]
    float* Ls = Vs + kC * kPad;           // [64][65]  L (strictly lower)
    float* Ts = Ls + kC * (kC + 1);       // [64][65]  T = (I + L)^-1
    float* g = Ts + kC * (kC + 1);        // [64] cumulative decay
    float* bt = g + kC;                   // [64] beta
    float* al = bt + kC;                  // [64] alpha
    const int tid = threadIdx.x;

    // rows of K, Q, V: 16 threads per row, 4 rows per pass of 64 threads ... 16 passes of 256
    for (int idx = tid; idx < kC * 16; idx += kPrepThreads) {
        const int t = idx / 16, p = idx % 16;
        const bool valid = t < len;
        const int64_t tok = static_cast<int64_t>(t0) + t;
        load_row_bf16(Ks + t * kPad, k + (tok * h_qk + jq) * kD, valid, p);
        load_row_bf16(Qs + t * kPad, q + (tok * h_qk + jq) * kD, valid, p);
        load_row_bf16(Vs + t * kPad, v + (tok * h_v + j) * kD, valid, p);
    }
    if (tid < kC) {
        const bool valid = tid < len;
        const int64_t tok = static_cast<int64_t>(t0) + tid;
        al[tid] = valid ? alpha[tok * h_v + j] : 1.f;
        bt[tid] = valid ? beta[tok * h_v + j] : 0.f;
    }
    __syncthreads();
    if (tid == 0) {
        float p = 1.f;
        for (int t = 0; t < kC; ++t) {
            p *= al[t];
            g[t] = p;
        }
    }
    __syncthreads();

    // L = strictly lower part of diag(beta) (g_t / g_s) K K^T; A^T[s][t] = (g_t / g_s) q_t . k_s
    float* atc = at + (static_cast<int64_t>(ch) * h_v + j) * kC * kC;
    for (int idx = tid; idx < kC * kC; idx += kPrepThreads) {
        const int t = idx / kC, s = idx % kC;
        float kk = 0.f, qk = 0.f;
        if (s <= t) {
            const float* kt = Ks + t * kPad;
            const float* qt = Qs + t * kPad;
            const float* ks = Ks + s * kPad;
#pragma unroll 8
            for (int c = 0; c < kD; ++c) {
                kk = fmaf(kt[c], ks[c], kk);
                qk = fmaf(qt[c], ks[c], qk);
            }
        }
        const float ratio = s <= t ? g[t] / g[s] : 0.f;
        Ls[t * (kC + 1) + s] = s < t ? bt[t] * ratio * kk : 0.f;
        atc[s * kC + t] = ratio * qk;
    }
    __syncthreads();

    // T = (I + L)^-1 by forward substitution, one row at a time (row t needs rows < t)
    for (int t = 0; t < kC; ++t) {
        if (tid < kC) {
            const int s = tid;
            float x = 0.f;
            if (s < t) {
                for (int m = s; m < t; ++m) x = fmaf(Ls[t * (kC + 1) + m], Ts[m * (kC + 1) + s], x);
                x = -x;
            } else if (s == t) {
                x = 1.f;
            }
            Ts[t * (kC + 1) + s] = x;
        }
        __syncthreads();
    }

    // W^T[c][t] = sum_{s<=t} T[t][s] beta_s g_s K[s][c];  U'^T[c][t] = sum_{s<=t} T[t][s] beta_s V[s][c]
    {
        const int t = tid % kC;
        const int cg = tid / kC;                  // 4 groups of 32 columns
        float* wtc = wt + (static_cast<int64_t>(ch) * h_v + j) * kD * kC;
        float* utc = ut + (static_cast<int64_t>(ch) * h_v + j) * kD * kC;
        for (int cc = 0; cc < 32; ++cc) {
            const int c = cg * 32 + cc;
            float w = 0.f, u = 0.f;
            for (int s = 0; s <= t; ++s) {
                const float ts = Ts[t * (kC + 1) + s] * bt[s];
                w = fmaf(ts * g[s], Ks[s * kPad + c], w);
                u = fmaf(ts, Vs[s * kPad + c], u);
            }
            wtc[c * kC + t] = w;
            utc[c * kC + t] = u;
        }
    }
    if (tid < kC) gam_out[(static_cast<int64_t>(ch) * h_v + j) * kC + tid] = g[tid];
}

// ---- per (sequence, value head, block of 16 value rows): the state scan over the chunks -----
constexpr int kScanThreads = 128;
constexpr size_t kScanSmem =
    sizeof(float) * (kRows * kD + kD * kC + kC * kC + 2 * kRows * kC + kD * (kC + 1) + kC * kD +
                     2 * kC);

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
    extern __shared__ float sm[];
    float* S = sm;                        // [16][128] state rows r0 .. r0+15
    float* Wt = S + kRows * kD;           // [128][64]
    float* At = Wt + kD * kC;             // [64 s][64 t]
    float* Up = At + kC * kC;             // [16][64]  U' rows
    float* U = Up + kRows * kC;           // [16][64]  U rows
    float* Qt = U + kRows * kC;           // [128][65] Q transposed
    float* Kc = Qt + kD * (kC + 1);       // [64][128]
    float* g = Kc + kC * kD;              // [64]
    float* kf = g + kC;                   // [64] g_C / g_s
    const int tid = threadIdx.x;

    const int64_t sbase = ((static_cast<int64_t>(i) * h_v + j) * kD + r0) * kD;
    for (int e = tid; e < kRows * kD; e += kScanThreads) S[e] = s0 ? s0[sbase + e] : 0.f;

    const int32_t c_begin = chunk_offset[i], c_end = chunk_offset[i + 1];
    const int32_t seq_start = cu[i];
    for (int32_t ch = c_begin; ch < c_end; ++ch) {
        const int32_t t0 = seq_start + (ch - c_begin) * kC;
        const int32_t len = min(kC, cu[i + 1] - t0);
        __syncthreads();   // the previous chunk's readers are done with the tiles
        const int64_t cj = static_cast<int64_t>(ch) * h_v + j;
        {
            const float4* src = reinterpret_cast<const float4*>(wt + cj * kD * kC);
            for (int e = tid; e < kD * kC / 4; e += kScanThreads)
                reinterpret_cast<float4*>(Wt)[e] = __ldg(src + e);
            const float4* asrc = reinterpret_cast<const float4*>(at + cj * kC * kC);
            for (int e = tid; e < kC * kC / 4; e += kScanThreads)
                reinterpret_cast<float4*>(At)[e] = __ldg(asrc + e);
            const float4* usrc = reinterpret_cast<const float4*>(ut + (cj * kD + r0) * kC);
            for (int e = tid; e < kRows * kC / 4; e += kScanThreads)
                reinterpret_cast<float4*>(Up)[e] = __ldg(usrc + e);
            if (tid < kC) g[tid] = __ldg(gam + cj * kC + tid);
        }
        for (int idx = tid; idx < kC * 16; idx += kScanThreads) {
            const int t = idx / 16, p = idx % 16;
            const bool valid = t < len;
            const int64_t tok = static_cast<int64_t>(t0) + t;
            float f[8];
            const __nv_bfloat16* qsrc = q + (tok * h_qk + jq) * kD;
            const __nv_bfloat16* ksrc = k + (tok * h_qk + jq) * kD;
            if (valid) {
                const uint4 w = __ldg(reinterpret_cast<const uint4*>(qsrc) + p);
                const uint32_t u[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    f[2 * e] = __uint_as_float(u[e] << 16);
                    f[2 * e + 1] = __uint_as_float(u[e] & 0xFFFF0000u);
                }
            } else {
#pragma unroll
                for (int e = 0; e < 8; ++e) f[e] = 0.f;
            }
#pragma unroll
            for (int e = 0; e < 8; ++e) Qt[(p * 8 + e) * (kC + 1) + t] = f[e];
            load_row_bf16(Kc + t * kD, ksrc, valid, p);
        }
        __syncthreads();
        if (tid < kC) kf[tid] = g[kC - 1] / g[tid];

        // U[r][t] = U'[r][t] - sum_c W[t][c] S[r][c]
        const int t = tid % kC;
        const int rg = tid / kC;                  // rows rg*8 .. rg*8+7
        {
            float acc[8];
#pragma unroll
            for (int r = 0; r < 8; ++r) acc[r] = Up[(rg * 8 + r) * kC + t];
            for (int c = 0; c < kD; ++c) {
                const float w = Wt[c * kC + t];
#pragma unroll
                for (int r = 0; r < 8; ++r) acc[r] = fmaf(-w, S[(rg * 8 + r) * kD + c], acc[r]);
            }
#pragma unroll
            for (int r = 0; r < 8; ++r) U[(rg * 8 + r) * kC + t] = acc[r];
        }
        __syncthreads();

        // O[t][r] = scale (g_t sum_c Q[t][c] S[r][c] + sum_{s<=t} A[t][s] U[r][s])
        {
            float qs[8], au[8];
#pragma unroll
            for (int r = 0; r < 8; ++r) qs[r] = au[r] = 0.f;
            for (int c = 0; c < kD; ++c) {
                const float qv = Qt[c * (kC + 1) + t];
#pragma unroll
                for (int r = 0; r < 8; ++r) qs[r] = fmaf(qv, S[(rg * 8 + r) * kD + c], qs[r]);
            }
            for (int s = 0; s <= t; ++s) {
                const float a = At[s * kC + t];
#pragma unroll
                for (int r = 0; r < 8; ++r) au[r] = fmaf(a, U[(rg * 8 + r) * kC + s], au[r]);
            }
            if (t < len) {
                const int64_t tok = static_cast<int64_t>(t0) + t;
                __nv_bfloat16* dst = o + (tok * h_v + j) * kD + r0 + rg * 8;
                uint32_t packed[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const float x0 = scale * fmaf(g[t], qs[2 * e], au[2 * e]);
                    const float x1 = scale * fmaf(g[t], qs[2 * e + 1], au[2 * e + 1]);
                    const __nv_bfloat162 h = __floats2bfloat162_rn(x0, x1);
                    packed[e] = *reinterpret_cast<const uint32_t*>(&h);
                }
                *reinterpret_cast<uint4*>(dst) = make_uint4(packed[0], packed[1], packed[2],
                                                            packed[3]);
            }
        }
        __syncthreads();   // every reader of S is done before the update

        // H_next[r][c] = g_C H[r][c] + sum_s U[r][s] (g_C / g_s) K[s][c]
        {
            const int c = tid;                    // 128 threads, one column each
            const float gC = g[kC - 1];
            float acc[kRows];
#pragma unroll
            for (int r = 0; r < kRows; ++r) acc[r] = gC * S[r * kD + c];
            for (int s = 0; s < kC; ++s) {
                const float kv = kf[s] * Kc[s * kD + c];
#pragma unroll
                for (int r = 0; r < kRows; ++r) acc[r] = fmaf(U[r * kC + s], kv, acc[r]);
            }
#pragma unroll
            for (int r = 0; r < kRows; ++r) S[r * kD + c] = acc[r];
        }
    }
    __syncthreads();
    if (s_final)
        for (int e = tid; e < kRows * kD; e += kScanThreads) s_final[sbase + e] = S[e];
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
