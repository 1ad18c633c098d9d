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
// depend on the chunk alone (gdn_prepare_kernel, all chunks in parallel).  The scan over a
// sequence's chunks (gdn_scan_kernel) then computes, with g_C the chunk's last decay,
//     U  = U' - W H0^T                         (the chunk's true updates)
//     U~ = diag(g_C / g) U                     (each update decayed to the chunk's end)
//     O  = scale (diag(g) Q H0^T + A' U~),     A'[t][s] = (g_t / g_C) (q_t . k_s) for s <= t
//     H_next = g_C H0 + U~^T K
// (A' U~ equals the intra-chunk attention term sum_{s<=t} (g_t / g_s) (q_t . k_s) u_s).  Every
// value row of H evolves on its own, so the scan splits a head's dv rows over several CTAs.
//
// Precision.  The products run on the tensor cores as bfloat16 x bfloat16 -> fp32 (exact
// products).  q and k are bfloat16 already; an fp32 operand x is carried as three bfloat16
// pieces x0 + x1 + x2 (x0 = bf16(x), x1 = bf16(x - x0), x2 = bf16(x - x0 - x1): |x - x0 - x1 -
// x2| <= 2^-27 |x|), and a product of two such operands keeps the six terms of order <= 2, so
// the state path stays at fp32 accuracy.  The output path (A' U~), which ends in a bfloat16
// result, keeps two pieces of each and three terms (relative error about 2^-16).
//
// A sequence's last chunk may be short: its missing tokens are read as q = k = v = 0,
// alpha = 1, beta = 0 (the page's rule for packed tails), which leaves the state and the valid
// outputs unchanged.  Non-product arithmetic is fp32; q, k, v and o are bfloat16.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <cstdarg>
#include <cstdint>
#include <cstdlib>
#include <atomic>
#include <cstdio>
#include <mutex>
#include <string>
#include <type_traits>

#include "../../include/gdn.h"
#include "desc.h"
#include "gdn_offsets.h"
#include "ptx.cuh"

namespace {

constexpr int kC = 64;          // tokens per chunk
constexpr int kD = 128;         // head dimension (dk = dv)
constexpr int kRows = 16;       // value rows of the state per scan CTA
constexpr int kMaxDevices = 64;  // device ordinals the per-device set-up covers

thread_local std::string t_gdn_error;
std::atomic<uint64_t> g_gdn_wait_ns{2000000000ull};   // limit of one wait for a chunk's loads
std::atomic<uint32_t> g_gdn_fault{0};                 // testing hook (gdn_set_fault_injection)
std::atomic<int> g_gdn_scan{GDN_SCAN_AUTO};           // scan kernel (gdn_set_scan_kernel)

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

// Workspace layout (all offsets 256-byte aligned), per chunk cj = chunk * h_v + value head:
//   wp   bf16 [cj][3][64][128]  W in three pieces, rows t, columns c
//   ap   bf16 [cj][2][64][64]   A' in two pieces, rows t, columns s (zero for s > t)
//   ut   f32  [cj][128][64]     U'^T, rows v, columns t
//   gam  f32  [cj][128]         g_t (t < 64), then g_C / g_t
// plus a status word the scan sets when a wait for its loads runs out (gdn_check_status), the
// scan's work-item counter and the order in which it takes the sequences (with their chunk and
// token ranges).
struct WsLayout {
    size_t status, counter, order, seqinfo, chunk_offset, n_chunks, chunks, wp, ap, ut, gam, total;
};

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

WsLayout layout_for(int64_t T, int64_t n, int64_t h_v)
{
    const size_t mc = static_cast<size_t>(max_chunks_for(T, n));
    const size_t cj = mc * static_cast<size_t>(h_v);
    WsLayout l{};
    size_t o = 0;
    l.status = o;       o = align256(o + sizeof(uint32_t));
    l.counter = o;      o = align256(o + sizeof(uint32_t));
    l.order = o;        o = align256(o + sizeof(int32_t) * static_cast<size_t>(n));
    l.seqinfo = o;      o = align256(o + sizeof(int4) * static_cast<size_t>(n));
    l.chunk_offset = o; o = align256(o + sizeof(int32_t) * static_cast<size_t>(n + 1));
    l.n_chunks = o;     o = align256(o + sizeof(int32_t));
    l.chunks = o;       o = align256(o + sizeof(int4) * mc);
    l.wp = o;           o = align256(o + sizeof(__nv_bfloat16) * cj * 3 * kC * kD);
    l.ap = o;           o = align256(o + sizeof(__nv_bfloat16) * cj * 2 * kC * kC);
    l.ut = o;           o = align256(o + sizeof(float) * cj * kD * kC);
    l.gam = o;          o = align256(o + sizeof(float) * cj * 2 * kC);
    l.total = o;
    return l;
}

// Programmatic dependent launch.  A kernel launched with programmatic stream serialization may
// start while the kernel before it on the stream still runs; grid_dep_wait() returns once that
// kernel has completed and its memory writes are visible (at once when the launch had no such
// dependency).  grid_dep_launch() lets the next kernel of the stream start early; it launches
// once every CTA of this grid has called it or exited.
__device__ __forceinline__ void grid_dep_wait()
{
    asm volatile("griddepcontrol.wait;" ::: "memory");
}
__device__ __forceinline__ void grid_dep_launch()
{
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ---- chunk list: per sequence, ceil(len / 64) chunks, numbered in sequence order -------------
// The offsets are checked first (non-decreasing, from 0 to total_tokens).  Offsets that break
// that contract are refused: the status word gets kStatusBadOffsets and every sequence is listed
// as empty (no chunk, no token), so the prepare kernel does nothing and the scan only passes the
// states through.  Either way this kernel writes only the workspace's tables, at indices bounded
// by n_seqs and max_chunks.
__global__ void gdn_chunk_list_kernel(const int32_t* __restrict__ cu, int32_t n_seqs,
                                      int32_t total_tokens,
                                      int32_t* __restrict__ chunk_offset, int4* __restrict__ chunks,
                                      int32_t max_chunks, int32_t* __restrict__ n_chunks,
                                      uint32_t* __restrict__ status, int32_t* __restrict__ order,
                                      int4* __restrict__ seqinfo, uint32_t* __restrict__ counter)
{
    // The call's first kernel, launched programmatically: it waits for whatever ran before it
    // on the stream (which may have written cu_seqlens, or still read the workspace's tables)
    // before it reads or writes anything, and only then lets the prepare kernel start.
    grid_dep_wait();
    grid_dep_launch();   // the prepare kernel may set itself up meanwhile
    bool bad = false;
    for (int32_t i = threadIdx.x; i < n_seqs; i += blockDim.x)
        bad |= !gdn::offsets_pair_ok(cu[i], cu[i + 1]);
    if (threadIdx.x == 0) bad |= !gdn::offsets_ends_ok(cu[0], cu[n_seqs], total_tokens);
    bad = __syncthreads_or(bad);
    if (threadIdx.x == 0) {
        *status = bad ? gdn::kStatusBadOffsets : 0u;   // this call's kernels report into it
        *counter = 0u;                                 // the scan's work-item counter
    }
    if (bad) {   // refused: every sequence empty, in index order
        for (int32_t i = threadIdx.x; i <= n_seqs; i += blockDim.x) chunk_offset[i] = 0;
        for (int32_t i = threadIdx.x; i < n_seqs; i += blockDim.x) {
            order[i] = i;
            seqinfo[i] = make_int4(0, 0, 0, 0);
        }
        if (threadIdx.x == 0) *n_chunks = 0;
        return;
    }
    __shared__ int32_t scan[1024];
    __shared__ int32_t ncs[1024];
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
        ncs[threadIdx.x] = nc;
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
    __syncthreads();   // chunk_offset complete
    // The scan takes sequences longest first (fewer idle SMs at the end): order[rank] = sequence,
    // ranked by chunk count, ties by index, and seqinfo[rank] = {first chunk, end chunk, first
    // token, end token}.  Up to 1024 sequences (the counts are still in ncs); beyond that, in
    // index order.
    for (int32_t i = threadIdx.x; i < n_seqs; i += blockDim.x) {
        int32_t rank = i;
        if (n_seqs <= static_cast<int32_t>(blockDim.x)) {
            const int32_t mine = ncs[i];
            rank = 0;
            for (int32_t o = 0; o < n_seqs; ++o) rank += ncs[o] > mine || (ncs[o] == mine && o < i);
        }
        order[rank] = i;
        seqinfo[rank] = make_int4(chunk_offset[i], chunk_offset[i + 1], cu[i], cu[i + 1]);
    }
}

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
__device__ __forceinline__ void mma_bf16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                         uint32_t b1)
{
    mma_bf16(d, a[0], a[1], a[2], a[3], b0, b1);
}

// ldmatrix / stmatrix of 8 x 8 blocks of 16-bit elements; lane l supplies the shared address of
// row l % 8 of block l / 8.
__device__ __forceinline__ uint32_t smem_u32(const void* p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void ldsm_x4(uint32_t (&r)[4], uint32_t addr)
{
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]) : "r"(addr));
}
__device__ __forceinline__ void ldsm_x2(uint32_t (&r)[2], uint32_t addr)
{
    asm volatile("ldmatrix.sync.aligned.m8n8.x2.shared.b16 {%0, %1}, [%2];"
                 : "=r"(r[0]), "=r"(r[1]) : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_trans(uint32_t (&r)[4], uint32_t addr)
{
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]) : "r"(addr));
}
__device__ __forceinline__ void stsm_x2_trans(uint32_t addr, uint32_t r0, uint32_t r1)
{
    asm volatile("stmatrix.sync.aligned.m8n8.x2.trans.shared.b16 [%0], {%1, %2};"
                 ::"r"(addr), "r"(r0), "r"(r1) : "memory");
}

// Three bfloat16 pieces of x (x0 + x1 + x2 within 2^-27 |x|), packed for two values a (low
// half) and b (high half) of one fragment register.
struct Pieces3 { uint32_t p[3]; };
__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi)
{
    const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<const uint32_t*>(&v);
}
__device__ __forceinline__ Pieces3 split3(float a, float b)
{
    Pieces3 r;
    const __nv_bfloat162 v0 = __floats2bfloat162_rn(a, b);
    const float a1 = a - __low2float(v0), b1 = b - __high2float(v0);
    const __nv_bfloat162 v1 = __floats2bfloat162_rn(a1, b1);
    const float a2 = a1 - __low2float(v1), b2 = b1 - __high2float(v1);
    r.p[0] = *reinterpret_cast<const uint32_t*>(&v0);
    r.p[1] = *reinterpret_cast<const uint32_t*>(&v1);
    r.p[2] = pack_bf16(a2, b2);
    return r;
}

// Shared-memory tiles of bfloat16 rows stored in 16-byte granules, granule index XOR (row % 8):
// the eight rows an ldmatrix / stmatrix block touches then fall in eight different bank groups.
// Rows of 128 elements (256 bytes) and of 64 elements (128 bytes).
__device__ __forceinline__ uint32_t sw256(int row, int col)
{
    return static_cast<uint32_t>(row * 256 + (((col >> 3) ^ (row & 7)) * 16) + (col & 7) * 2);
}
__device__ __forceinline__ uint32_t sw128(int row, int col)
{
    return static_cast<uint32_t>(row * 128 + (((col >> 3) ^ row) & 7) * 16 + (col & 7) * 2);
}

// Byte offset of element (row, col) in a 128-column bf16 tile that TMA wrote as two 64-column
// halves of `rows` 128-byte rows each, 128-byte swizzle (16-byte granule g of row r at g ^ (r % 8)).
__device__ __forceinline__ uint32_t tsw(int row, int col, int rows)
{
    return static_cast<uint32_t>((col >> 6) * rows * 128 + row * 128 +
                                 ((((col >> 3) & 7) ^ (row & 7)) << 4) + (col & 7) * 2);
}

// Byte offset of element (row, col) in a 64-column fp32 tile that TMA reads or writes as two
// 32-column halves of 128 rows of 128 bytes each, 128-byte swizzle.
__device__ __forceinline__ uint32_t tsw32(int row, int col)
{
    return static_cast<uint32_t>((col >> 5) * 128 * 128 + row * 128 +
                                 ((((col >> 2) & 7) ^ (row & 7)) << 4) + (col & 3) * 4);
}
__device__ __forceinline__ void st_shared_u32(uint32_t addr, uint32_t v)
{
    asm volatile("st.shared.b32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}
__device__ __forceinline__ void st_shared_f32(uint32_t addr, float v)
{
    asm volatile("st.shared.f32 [%0], %1;" ::"r"(addr), "f"(v) : "memory");
}

// ---- per (chunk, value head): W, U'^T, A' and the cumulative decays ----------------------------
// K, Q, V of the chunk arrive by TMA as 128-byte-swizzled bf16 tiles.  Products K K^T and Q K^T
// run on the tensor cores (bf16 operands, exact products).  T = (I + L)^-1 is then built in the
// page's doubling stages: the eight 8 x 8 diagonal blocks by substitution, then for block sizes
// b = 8, 16, 32 each pair of neighbouring inverted blocks [A 0; C B] becomes
// [A^-1 0; -B^-1 C A^-1  B^-1] (fp32 dot products for b = 8; for b = 16 and 32 tensor-core
// products of three-piece bfloat16 operands, at fp32 accuracy).  Finally W = T diag(beta g) K and
// U' = T diag(beta) V run on the tensor cores: T diag(.) as three bfloat16 pieces against the
// exact bfloat16 K or V, the three products keeping fp32 accuracy.
constexpr int kRowA = 72;      // padded bf16 rows of A' staging (144 bytes)
constexpr int kRowL = 68;      // padded fp32 rows of L and T (272 bytes)
constexpr int kRowY = 36;      // fp32 rows of the doubling scratch (144 bytes: 16-byte aligned)
constexpr int kPrepThreads = 256;
// K, Q, V: 128-byte-swizzled TMA tiles (two 64-column halves of 64 rows) at a 1024-byte-aligned
// base, then the A' staging, L, T and the per-token vectors, then the load barrier.
constexpr uint32_t kPrepTile = 2 * kC * 128;   // one of K, Q, V
constexpr size_t kPrepSmem = 3 * kPrepTile + sizeof(__nv_bfloat16) * 2 * kC * kRowA +
                             sizeof(float) * (2 * kC * kRowL + 4 * kC) + 16 + 1024;
// A prepare grid of no more CTAs than SMs asks for this much shared memory instead: more than
// half of what an SM has, so that no SM runs two of its CTAs while another runs none.
constexpr size_t kPrepSpreadSmem = 120 * 1024;
static_assert(kPrepSpreadSmem >= kPrepSmem && 2 * (kPrepSpreadSmem + 1024) > 233472,
              "one prepare CTA per SM at the spread size");
static_assert(sizeof(__nv_bfloat16) * 2 * kC * kRowA >= sizeof(float) * 32 * kRowY,
              "the doubling scratch reuses the A' staging");
static_assert(3 * kPrepTile == 3 * kC * kD * 2, "W's three pieces are staged over K, Q and V");
static_assert(sizeof(float) * kD * kC <=
                  sizeof(__nv_bfloat16) * 2 * kC * kRowA + sizeof(float) * kC * kRowL,
              "U'^T is staged over the A' staging and L, before T");

// One doubling stage of T = (I + L)^-1 for block size b (T holds the inverted b x b diagonal
// blocks; their upper parts are zero): for each pair [A 0; C B] at rows / columns r0 = 2 p b, the
// lower-left block of the inverse is -B^-1 (C A^-1).  The 32 rows (p, i) of each product take
// 8 threads apiece, each thread U = b / 8 consecutive columns (one vector load per operand row),
// full-length (zero-padded) dot products.
template <int b>
__device__ __forceinline__ void invert_doubling_stage(const float* Ls, float* Ts, float* Yb, int tid)
{
    constexpr int U = b / 8;
    using Vec = typename std::conditional<U == 4, float4, typename std::conditional<U == 2, float2,
                                                                                    float>::type>::type;
    const int row = tid >> 3, l8 = tid & 7;
    const int p = row / b, i = row % b, r0 = 2 * p * b;
    const auto fma_vec = [](float c, const Vec& x, float (&acc)[U]) {
        const float* xv = reinterpret_cast<const float*>(&x);
#pragma unroll
        for (int u = 0; u < U; ++u) acc[u] = fmaf(c, xv[u], acc[u]);
    };
    float acc[U];
#pragma unroll
    for (int u = 0; u < U; ++u) acc[u] = 0.f;
    {   // Y = C A^-1
        const float* crow = Ls + (r0 + b + i) * kRowL + r0;
        const float* acol = Ts + r0 * kRowL + r0 + U * l8;
#pragma unroll
        for (int m = 0; m < b; ++m)
            fma_vec(crow[m], *reinterpret_cast<const Vec*>(acol + m * kRowL), acc);
        *reinterpret_cast<Vec*>(Yb + row * kRowY + U * l8) = *reinterpret_cast<const Vec*>(acc);
    }
    __syncthreads();
#pragma unroll
    for (int u = 0; u < U; ++u) acc[u] = 0.f;
    {   // lower-left block = -B^-1 Y
        const float* brow = Ts + (r0 + b + i) * kRowL + r0 + b;
        const float* ycol = Yb + p * b * kRowY + U * l8;
#pragma unroll
        for (int m = 0; m < b; ++m)
            fma_vec(brow[m], *reinterpret_cast<const Vec*>(ycol + m * kRowY), acc);
#pragma unroll
        for (int u = 0; u < U; ++u) acc[u] = -acc[u];
        *reinterpret_cast<Vec*>(Ts + (r0 + b + i) * kRowL + r0 + U * l8) =
            *reinterpret_cast<const Vec*>(acc);
    }
    __syncthreads();
}

// The same doubling stage on the tensor cores, for b = 16 and 32: both products of a pair run as
// mma.sync m16n8k16 with each fp32 operand split into three bfloat16 pieces, keeping the six
// piece products above 2^-16 of the leading one (so the sum keeps fp32 accuracy).  Warp w owns
// output tile w of the stage: (pair, 16-row tile, 8-column tile); with b = 16 the four tiles
// leave warps 4-7 idle.  Y goes through the scratch rows as in the scalar stage.
template <int b>
__device__ __forceinline__ void invert_doubling_stage_tc(const float* Ls, float* Ts, float* Yb,
                                                         int tid)
{
    static_assert(b == 16 || b == 32, "tensor-core doubling stages are 16 and 32 wide");
    constexpr int kNT = b / 8;                 // 8-column tiles per pair
    constexpr int kTiles = (kC / (2 * b)) * (b / 16) * kNT;
    const int warp = tid / 32, lane = tid % 32;
    const int gq = lane >> 2, tg = lane & 3;
    const bool active = warp < kTiles;
    const int p = warp / ((b / 16) * kNT), mt = (warp / kNT) % (b / 16), nt = warp % kNT;
    const int r0 = 2 * p * b;
    // d = X Z over k = 0 .. b-1 for the warp's tile: X row-major fp32 (row stride xs), Z fp32
    // read as Z[k][n] (row stride zs).  The piece products of each order (i + j = 0, 1, 2) have
    // an accumulator of their own, so that no more than six MMAs wait on one another; the
    // smaller orders are added first.
    const auto product = [&](float (&d)[4], const float* X, int xs, const float* Z, int zs) {
        float e[3][4] = {};
#pragma unroll
        for (int kk = 0; kk < b / 16; ++kk) {
            const float* x0 = X + (16 * mt + gq) * xs + 16 * kk + 2 * tg;
            const float2 v00 = *reinterpret_cast<const float2*>(x0);
            const float2 v10 = *reinterpret_cast<const float2*>(x0 + 8 * xs);
            const float2 v01 = *reinterpret_cast<const float2*>(x0 + 8);
            const float2 v11 = *reinterpret_cast<const float2*>(x0 + 8 * xs + 8);
            const float* z0 = Z + (16 * kk + 2 * tg) * zs + 8 * nt + gq;
            const Pieces3 a0 = split3(v00.x, v00.y), a1 = split3(v10.x, v10.y);
            const Pieces3 a2 = split3(v01.x, v01.y), a3 = split3(v11.x, v11.y);
            const Pieces3 b0 = split3(z0[0], z0[zs]), b1 = split3(z0[8 * zs], z0[9 * zs]);
            // pieces (i, j) with i + j <= 2
#pragma unroll
            for (int i = 0; i < 3; ++i)
#pragma unroll
                for (int j = 0; i + j < 3; ++j)
                    mma_bf16(e[i + j], a0.p[i], a1.p[i], a2.p[i], a3.p[i], b0.p[j], b1.p[j]);
        }
#pragma unroll
        for (int r = 0; r < 4; ++r) d[r] = (e[2][r] + e[1][r]) + e[0][r];
    };
    if (active) {   // Y = C A^-1
        float d[4];
        product(d, Ls + (r0 + b) * kRowL + r0, kRowL, Ts + r0 * kRowL + r0, kRowL);
        float* y = Yb + (p * b + 16 * mt + gq) * kRowY + 8 * nt + 2 * tg;
        *reinterpret_cast<float2*>(y) = make_float2(d[0], d[1]);
        *reinterpret_cast<float2*>(y + 8 * kRowY) = make_float2(d[2], d[3]);
    }
    __syncthreads();
    if (active) {   // lower-left block = -B^-1 Y
        float d[4];
        product(d, Ts + (r0 + b) * kRowL + r0 + b, kRowL, Yb + p * b * kRowY, kRowY);
        float* x = Ts + (r0 + b + 16 * mt + gq) * kRowL + r0 + 8 * nt + 2 * tg;
        *reinterpret_cast<float2*>(x) = make_float2(-d[0], -d[1]);
        *reinterpret_cast<float2*>(x + 8 * kRowL) = make_float2(-d[2], -d[3]);
    }
    __syncthreads();
}

__global__ void __launch_bounds__(kPrepThreads, 2)
    gdn_prepare_kernel(const __grid_constant__ CUtensorMap map_q,
                       const __grid_constant__ CUtensorMap map_k,
                       const __grid_constant__ CUtensorMap map_v,
                       const __grid_constant__ CUtensorMap map_w,
                       const __grid_constant__ CUtensorMap map_ut, const float* __restrict__ alpha,
                       const float* __restrict__ beta, const int4* __restrict__ chunks,
                       const int32_t* __restrict__ n_chunks, int32_t h_v, int32_t qgroup,
                       int32_t kgroup, int32_t clear_status, __nv_bfloat16* __restrict__ ap,
                       float* __restrict__ gam_out, int32_t single_T,
                       const int32_t* __restrict__ cu, uint32_t* __restrict__ status,
                       uint32_t* __restrict__ counter, uint64_t wait_ns, int32_t first_in_call)
{
    const int32_t ch = blockIdx.x;
    const int32_t j = blockIdx.y;
    // This kernel may start while the kernel before it on the stream (the chunk list, or the
    // previous pass's scan) still runs.  Until grid_dep_wait() it reads only the call's inputs
    // (q, k, v, alpha, beta); the chunk list, the workspace and the counter wait for it.  Every
    // CTA passes grid_dep_wait() before it exits.  As a call's first kernel (one sequence, first
    // pass) it waits before anything: the kernel before it may be the previous call's scan, or
    // whatever wrote this call's inputs; and the scan may start only after that wait (it reads
    // its initial state early, which may be the previous call's final state).
    if (first_in_call) grid_dep_wait();
    grid_dep_launch();   // the scan may set itself up meanwhile
    // one sequence (single_T >= 0): chunk ch covers tokens 64 ch .. (no chunk list is built;
    // the first pass of a call, past its wait for everything before it, checks that the
    // offsets are [0, single_T] and sets the call's status word here, and offsets that are not
    // leave every chunk undone); otherwise the chunk list says
    int32_t t0, len;
    if (single_T >= 0) {
        const bool ok = gdn::offsets_single_ok(cu[0], cu[1], single_T);
        if (ch == 0 && j == 0 && threadIdx.x == 0 && clear_status)
            *status = ok ? 0u : gdn::kStatusBadOffsets;
        t0 = ch * kC;
        if (!ok || t0 >= single_T) {
            grid_dep_wait();
            return;
        }
        len = min(kC, single_T - t0);
    } else {
        grid_dep_wait();
        if (ch >= *n_chunks) return;
        const int4 info = chunks[ch];
        t0 = info.y;
        len = info.z;
    }
    const int32_t jq = j / qgroup, jk = j / kgroup;   // query / key head of state head j
    const int64_t cj = static_cast<int64_t>(ch) * h_v + j;
    const int tid = threadIdx.x;
    // alpha and beta first: their latency overlaps the tile loads
    float a_in = 1.f, b_in = 0.f;
    if (tid < kC && tid < len) {
        const int64_t tok = static_cast<int64_t>(t0) + tid;
        a_in = alpha[tok * h_v + j];
        b_in = beta[tok * h_v + j];
    }
    extern __shared__ __align__(16) uint8_t smraw[];
    const uint32_t raw = smem_u32(smraw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t* gbase = smraw + (base - raw);
    const uint32_t kb_s = base, qb_s = base + kPrepTile, vb_s = base + 2 * kPrepTile;
    const uint32_t ut_s = base + 3 * kPrepTile;   // U'^T staging at the end (A' staging and L)
    __nv_bfloat16* Ap = reinterpret_cast<__nv_bfloat16*>(gbase + 3 * kPrepTile);   // [2][64][72]
    float* Yb = reinterpret_cast<float*>(Ap);                         // [32][33], after A' is out
    float* Ls = reinterpret_cast<float*>(Ap + 2 * kC * kRowA);       // [64][68] L, strictly lower
    float* Ts = Ls + kC * kRowL;                                      // [64][68] T = (I + L)^-1
    float* g = Ts + kC * kRowL;
    float* bt = g + kC;
    float* bg = bt + kC;
    float* al = bg + kC;
    const uint32_t bar = smem_u32(al + kC);

    // K, Q, V rows by TMA (two 64-column halves each).  Rows past the chunk's end read the next
    // sequence's tokens (zeros past the last token); their beta is 0, which zeroes their rows of
    // L, W and U', and A' keeps only s <= t.
    if (tid == 0) {
        gf16::mbar_init(bar, 1);
        gf16::fence_mbarrier_init();
        gf16::mbar_arrive_expect_tx(bar, 3 * kPrepTile);
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            gf16::tma_load_3d(kb_s + h * kC * 128, &map_k, bar, 64 * h, jk, t0);
            gf16::tma_load_3d(qb_s + h * kC * 128, &map_q, bar, 64 * h, jq, t0);
            gf16::tma_load_3d(vb_s + h * kC * 128, &map_v, bar, 64 * h, j, t0);
        }
    }
    for (int e = tid; e < kC * kRowL; e += kPrepThreads) Ts[e] = 0.f;   // upper blocks stay zero
    // the six 16 x 16 tiles of A' above the diagonal, both pieces: zero (16-byte stores)
    for (int e = tid; e < 2 * 6 * 32; e += kPrepThreads) {
        // upper tile u: row block 0, 0, 0, 1, 1, 2 and column block 1, 2, 3, 2, 3, 3 (4 bits each)
        constexpr int kUpper = 0x123233;
        const int pc = e / 192, u = (e % 192) / 32, r = (e % 32) / 2, hf = e % 2;
        const int mi = u < 3 ? 0 : (u < 5 ? 1 : 2);
        const int ni = (kUpper >> (4 * (5 - u))) & 15;
        *reinterpret_cast<int4*>(Ap + pc * kC * kRowA + (16 * mi + r) * kRowA + 16 * ni + 8 * hf) =
            make_int4(0, 0, 0, 0);
    }
    if (tid < kC) {
        al[tid] = a_in;
        bt[tid] = b_in;
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
        al[2 * tid] = 1.f / (before * a0);   // from here on al holds 1 / g
        al[2 * tid + 1] = 1.f / p;
    }
    {
        const bool ok = gf16::mbar_wait(bar, 0, nullptr, wait_ns);
        if (__syncthreads_or(!ok)) {   // the tiles never landed: report and stop
            if (tid == 0) atomicOr(status, gdn::kStatusTimeout);
            grid_dep_wait();
            return;
        }
    }
    if (tid < kC) bg[tid] = bt[tid] * g[tid];

    // K K^T and Q K^T on the tensor cores: mma.sync m16n8k16 with bf16 operands (exact products,
    // fp32 sums).  Only the ten 16 x 16 tiles on or below the diagonal are needed (L is strictly
    // lower, A' keeps s <= t; the six upper A' tiles were zeroed above).  Warps 0 and 1 take two
    // tiles of row block 3 each, the others one tile, so that each scheduler's two warps (w and
    // w + 4) carry three or two tiles.
    {
        const int warp = tid / 32, lane = tid % 32;
        const int gq = lane >> 2, tg = lane & 3;
        // per warp (4 bits each, warp 0 first): row block 3, 3, 2, 2, 2, 1, 1, 0 and first
        // column block 0, 2, 0, 1, 2, 0, 1, 0
        constexpr int kMi = 0x33222110, kNi = 0x02012010;
        const int m0 = 16 * ((kMi >> (4 * (7 - warp))) & 15);
        const int nb = 16 * ((kNi >> (4 * (7 - warp))) & 15);
        const int ntiles = warp < 2 ? 2 : 1;
        float kk[4][4] = {}, qk[4][4] = {};
        const int lr = lane & 7, lb = lane >> 3;
#pragma unroll
        for (int k0 = 0; k0 < kD; k0 += 16) {
            // A fragments: rows m0 + (lane % 16), columns k0 + 8 (lane / 16)
            uint32_t ka[4], qa[4];
            const uint32_t aoff = tsw(m0 + (lane & 15), k0 + 8 * (lane >> 4), kC);
            ldsm_x4(ka, kb_s + aoff);
            ldsm_x4(qa, qb_s + aoff);
#pragma unroll
            for (int np = 0; np < 2; ++np) {
                if (np >= ntiles) break;
                // B fragments of n-tiles 2 np, 2 np + 1: k rows n0 + lr, columns k0 + 8 (lb % 2)
                uint32_t kb4[4];
                ldsm_x4(kb4, kb_s + tsw(nb + 16 * np + 8 * (lb >> 1) + lr, k0 + 8 * (lb & 1), kC));
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    mma_bf16(kk[2 * np + h], ka, kb4[2 * h], kb4[2 * h + 1]);
                    mma_bf16(qk[2 * np + h], qa, kb4[2 * h], kb4[2 * h + 1]);
                }
            }
        }
        const float inv_gc = 1.f / g[kC - 1];
#pragma unroll
        for (int nt = 0; nt < 4; ++nt) {
            if (nt >= 2 * ntiles) break;
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int t = m0 + gq + 8 * h;
                const int s = nb + 8 * nt + 2 * tg;
                float av[2];
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    Ls[t * kRowL + s + e] = s + e < t ? bt[t] * (g[t] * al[s + e]) * kk[nt][2 * h + e] : 0.f;
                    av[e] = s + e <= t ? (g[t] * inv_gc) * qk[nt][2 * h + e] : 0.f;
                }
                const Pieces3 pa = split3(av[0], av[1]);
                *reinterpret_cast<uint32_t*>(Ap + t * kRowA + s) = pa.p[0];
                *reinterpret_cast<uint32_t*>(Ap + kC * kRowA + t * kRowA + s) = pa.p[1];
            }
        }
    }
    __syncthreads();

    // From here on the workspace is written: the kernel before this one must have finished
    // with it (the previous pass's scan reads it and draws from the counter).
    grid_dep_wait();
    if (ch == 0 && j == 0 && tid == 0) *counter = 0u;   // the scan's work counter
    // A' pieces to global, 16-byte granules
    {
        __nv_bfloat16* apc = ap + cj * 2 * kC * kC;
        for (int e = tid; e < 2 * kC * 8; e += kPrepThreads) {
            const int p = e / (kC * 8), t = (e / 8) % kC, c8 = e % 8;
            *reinterpret_cast<int4*>(apc + (p * kC + t) * kC + c8 * 8) =
                *reinterpret_cast<const int4*>(Ap + (p * kC + t) * kRowA + c8 * 8);
        }
    }

    // ---- T = (I + L)^-1 in doubling stages ----
    // the eight 8 x 8 diagonal blocks, one column per thread by substitution
    if (tid < kC) {
        const int r0 = 8 * (tid >> 3), jj = tid & 7;
        float x[8];
#pragma unroll
        for (int m = 0; m < 8; ++m) {
            float acc = m == jj ? 1.f : 0.f;
#pragma unroll
            for (int n = 0; n < m; ++n) acc = fmaf(-Ls[(r0 + m) * kRowL + r0 + n], x[n], acc);
            x[m] = acc;
        }
#pragma unroll
        for (int m = 0; m < 8; ++m) Ts[(r0 + m) * kRowL + r0 + jj] = x[m];
    }
    __syncthreads();
    invert_doubling_stage<8>(Ls, Ts, Yb, tid);
    invert_doubling_stage_tc<16>(Ls, Ts, Yb, tid);
    invert_doubling_stage_tc<32>(Ls, Ts, Yb, tid);

    // ---- W = T diag(beta g) K (warps 0-3) and U' = T diag(beta) V (warps 4-7) ----
    // Warp w owns rows t of m-tile mt (the two halves take the tiles in opposite orders, so that
    // the two warps of a scheduler share 5 causal steps) and all 128 columns (16 n-tiles).
    {
        const int warp = tid / 32, lane = tid % 32;
        const int gq = lane >> 2, tg = lane & 3, lr = lane & 7, lb = lane >> 3;
        const int half = warp >> 2;
        const int mt = half ? 3 - (warp & 3) : (warp & 3);
        const float* sc = half ? bt : bg;
        const uint32_t src_s = half ? vb_s : kb_s;
        float acc[16][4];
#pragma unroll
        for (int n = 0; n < 16; ++n) acc[n][0] = acc[n][1] = acc[n][2] = acc[n][3] = 0.f;
        for (int kk = 0; kk <= mt; ++kk) {
            // A = T diag(sc) for rows 16 mt + gq (+8), columns 16 kk + 2 tg (+1, +8, +9), in pieces
            const int ta = 16 * mt + gq, sa = 16 * kk + 2 * tg;
            const float* T0 = Ts + ta * kRowL + sa;
            const float* T1 = T0 + 8 * kRowL;
            const float c0 = sc[sa], c1 = sc[sa + 1], c8 = sc[sa + 8], c9 = sc[sa + 9];
            const Pieces3 a0 = split3(T0[0] * c0, T0[1] * c1);
            const Pieces3 a1 = split3(T1[0] * c0, T1[1] * c1);
            const Pieces3 a2 = split3(T0[8] * c8, T0[9] * c9);
            const Pieces3 a3 = split3(T1[8] * c8, T1[9] * c9);
#pragma unroll
            for (int q = 0; q < 8; ++q) {
                // B = K or V rows s = 16 kk .. + 15, columns of n-tiles 2q and 2q+1 (ldmatrix .trans)
                uint32_t bfr[4];
                ldsm_x4_trans(bfr, src_s + tsw(16 * kk + lr + 8 * (lb & 1), 8 * (2 * q + (lb >> 1)), kC));
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const uint32_t b0 = bfr[2 * h], b1 = bfr[2 * h + 1];
#pragma unroll
                    for (int pc = 0; pc < 3; ++pc)
                        mma_bf16(acc[2 * q + h], a0.p[pc], a1.p[pc], a2.p[pc], a3.p[pc], b0, b1);
                }
            }
        }
        // Both results leave through shared memory and TMA stores: W as three bfloat16 pieces
        // [piece][t][c] over the K / Q / V tiles (two 64-column halves of 192 rows, 128-byte
        // swizzle), U'^T as fp32 [v][t] over the A' staging and L (two 32-token halves of 128
        // rows, 128-byte swizzle).  Each warp's 4-byte stores land in 32 distinct banks.
        const int t = 16 * mt + gq;
        __syncthreads();   // every warp is done reading K, V and T
        if (!half) {
#pragma unroll
            for (int n = 0; n < 16; ++n) {
                const int c = 8 * n + 2 * tg;
                const Pieces3 lo = split3(acc[n][0], acc[n][1]), hi = split3(acc[n][2], acc[n][3]);
#pragma unroll
                for (int pc = 0; pc < 3; ++pc) {
                    st_shared_u32(kb_s + tsw(pc * kC + t, c, 3 * kC), lo.p[pc]);
                    st_shared_u32(kb_s + tsw(pc * kC + t + 8, c, 3 * kC), hi.p[pc]);
                }
            }
        } else {
#pragma unroll
            for (int n = 0; n < 16; ++n) {
                const int v0 = 8 * n + 2 * tg;
                st_shared_f32(ut_s + tsw32(v0, t), acc[n][0]);
                st_shared_f32(ut_s + tsw32(v0 + 1, t), acc[n][1]);
                st_shared_f32(ut_s + tsw32(v0, t + 8), acc[n][2]);
                st_shared_f32(ut_s + tsw32(v0 + 1, t + 8), acc[n][3]);
            }
        }
        gf16::fence_proxy_async_smem();   // visible to the tensor-memory-access unit
        __syncthreads();
        if (tid == 0) {
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                gf16::tma_store_2d(&map_w, kb_s + h * 3 * kC * 128, 64 * h,
                                   static_cast<int32_t>(cj * 3 * kC));
                gf16::tma_store_2d(&map_ut, ut_s + h * kD * 128, 32 * h,
                                   static_cast<int32_t>(cj * kD));
            }
            gf16::bulk_commit_group();
        }
    }
    if (tid < kC) {
        gam_out[cj * 2 * kC + tid] = g[tid];
        gam_out[cj * 2 * kC + kC + tid] = g[kC - 1] / g[tid];
    }
    // The CTA's shared memory must outlive the stores' reads of it; their writes are complete
    // when the grid is (the next kernel reads them after grid_dep_wait()).
    if (tid == 0) gf16::bulk_wait_group_read<0>();
}

// ---- per (sequence, value head, block of 16 value rows): the state scan over the chunks -------
// Each chunk's operands are double-buffered in shared memory and arrive by TMA: while chunk c is
// computed, one thread has the tensor-memory-access unit bring chunk c + 1 (the W and A' pieces
// and the q / k rows as 128-byte-swizzled boxes, the block's U'^T rows and the decays as bulk
// copies), all completing on the stage's mbarrier.  Sixteen warps; each product runs on
// mma.sync m16n8k16 (bf16 -> fp32) with fragments loaded by ldmatrix.
//   phase 1   U = U' - W S^T and P = Q S^T: warp w owns tokens 16 (w % 4) .. + 15, state rows
//             8 ((w / 4) % 2) .. + 7 and half h = w / 8 of the key columns; the upper half's
//             partial U goes through shared memory to the lower half's warp, which forms
//             U~ = diag(g_C / g) U and stores it as pieces, [r][t]
//   phase 2   S_next^T = g_C S^T + K^T U~: warp w owns key columns 16 (w % 8) .. + 15 and state
//             rows 8 (w / 8) .. + 7; the fp32 state lives in these registers from chunk to
//             chunk, and its pieces go to shared memory, [r][c], for the next chunk's phase 1
//             O = scale (diag(g) P + A' U~): both warps of a phase-1 tile add their half of
//             diag(g) P and about half of the causal A' U~ steps; the lower warp's partial goes
//             through shared memory and the upper warp writes the sum to o at the start of the
//             next chunk (or after the last)
// Three barriers per chunk: U partials ready, U~ complete, state pieces complete and the next
// chunk's loads landed.
constexpr int kScanThreads = 512;
// shared-memory layout (offsets from a 1024-byte-aligned base)
constexpr uint32_t kStageBytes = 98304;               // TMA boxes of one chunk
constexpr uint32_t kOffW = 0;                         // W pieces: 2 column halves x 192 rows x 128 B
constexpr uint32_t kOffQ = 49152;                     // q: 2 halves x 64 rows x 128 B
constexpr uint32_t kOffK = 65536;                     // k: same
constexpr uint32_t kOffA = 81920;                     // A' pieces: 128 rows x 128 B
constexpr uint32_t kOffUp = 2 * kStageBytes;          // U'^T rows [stage][16][64] f32
constexpr uint32_t kOffG = kOffUp + 2 * kRows * kC * 4;      // [stage][g_t | g_C / g_t] f32
constexpr uint32_t kOffSp = kOffG + 2 * 2 * kC * 4;          // state pieces [3][16][128] bf16
constexpr uint32_t kOffUt = kOffSp + 3 * kRows * kD * 2;     // U~ pieces [3][16][64] bf16
constexpr uint32_t kOffPart = kOffUt + 3 * kRows * kC * 2;   // partial sums [8 warps][4][32] f32
constexpr uint32_t kOffBar = kOffPart + 8 * 4 * 32 * 4;      // two mbarriers
constexpr uint32_t kOffItem = kOffBar + 16;                  // the CTA's next item
constexpr uint32_t kStageTx = kStageBytes + kRows * kC * 4 + 2 * kC * 4;   // bytes per chunk
constexpr size_t kScanSmem = kOffItem + 16 + 1024;           // + slack to align the base
static_assert(kScanSmem <= 232448, "scan shared memory");


// Bulk (untiled) global -> shared copy completing on an mbarrier of this CTA.
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar)
{
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
                 ::"r"(dst), "l"(src), "r"(bytes), "r"(bar)
                 : "memory");
}

// One thread: announce the chunk's bytes on the stage barrier and start its loads.
__device__ __forceinline__ void scan_issue(uint32_t base, int s, uint32_t bar,
                                           const CUtensorMap* map_w, const CUtensorMap* map_a,
                                           const CUtensorMap* map_q, const CUtensorMap* map_k,
                                           const float* __restrict__ ut,
                                           const float* __restrict__ gam, int64_t cj, int32_t r0,
                                           int32_t t0, int32_t jq, int32_t jk)
{
    gf16::mbar_arrive_expect_tx(bar, kStageTx);
    const uint32_t st = base + s * kStageBytes;
    const int32_t yw = static_cast<int32_t>(cj * 3 * kC), ya = static_cast<int32_t>(cj * 2 * kC);
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        gf16::tma_load_2d(st + kOffW + h * 3 * kC * 128, map_w, bar, 64 * h, yw);
        gf16::tma_load_3d(st + kOffQ + h * kC * 128, map_q, bar, 64 * h, jq, t0);
        gf16::tma_load_3d(st + kOffK + h * kC * 128, map_k, bar, 64 * h, jk, t0);
    }
    gf16::tma_load_2d(st + kOffA, map_a, bar, 0, ya);
    bulk_g2s(base + kOffUp + s * kRows * kC * 4, ut + (cj * kD + r0) * kC, kRows * kC * 4, bar);
    bulk_g2s(base + kOffG + s * 2 * kC * 4, gam + cj * 2 * kC, 2 * kC * 4, bar);
}

// kMulti: a CTA may take more than one work item (more items than CTAs); without it every CTA
// runs exactly item blockIdx.x and the scheduling code drops out.
template <bool kMulti>
__global__ void __launch_bounds__(kScanThreads, 1)
    gdn_scan_kernel(const __grid_constant__ CUtensorMap map_w,
                    const __grid_constant__ CUtensorMap map_a,
                    const __grid_constant__ CUtensorMap map_q,
                    const __grid_constant__ CUtensorMap map_k, const int32_t* __restrict__ order,
                    const int4* __restrict__ seqinfo, uint32_t* __restrict__ counter,
                    int32_t n_items, const float* __restrict__ ut,
                    const float* __restrict__ gam, const float* __restrict__ s0,
                    float* __restrict__ s_final, __nv_bfloat16* __restrict__ o,
                    uint32_t* __restrict__ status, int32_t h_v, int32_t qgroup, int32_t kgroup,
                    int32_t o_tok, int32_t o_hmul, float scale,
                    uint64_t wait_ns, uint32_t fault, int32_t single_T,
                    const int32_t* __restrict__ cu)
{
    extern __shared__ __align__(16) uint8_t smraw[];
    const uint32_t raw = smem_u32(smraw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t* gbase = smraw + (base - raw);
    const float* upf = reinterpret_cast<const float*>(gbase + kOffUp);
    const float* gf = reinterpret_cast<const float*>(gbase + kOffG);
    float* part = reinterpret_cast<float*>(gbase + kOffPart);
    volatile int32_t* next_item = reinterpret_cast<volatile int32_t*>(gbase + kOffItem);
    const uint32_t sp_s = base + kOffSp, up_s = base + kOffUt, bar0 = base + kOffBar;
    const int tid = threadIdx.x;
    const int warp = tid / 32, lane = tid % 32;
    const int gq = lane >> 2, tg = lane & 3;
    const int lr = lane & 7, lb = lane >> 3;                    // ldmatrix row, block

    if (tid == 0) {
        gf16::mbar_init(bar0, 1);
        gf16::mbar_init(bar0 + 8, 1);
        gf16::fence_mbarrier_init();
    }

    // Work items are (sequence, value head, block of 16 state rows), numbered sequence-major in
    // the order `order` gives (longest sequences first); item q -> rank q / (8 h_v), head
    // (q / 8) % h_v, rows 16 (q % 8) ...  With G = gridDim.x, CTA b's first item is b and each
    // later one G + a value drawn from `counter` when the item before it starts (a
    // longest-processing-time schedule).  Thread 0 makes the draw as the item starts and
    // publishes it at the first chunk's middle barrier; the next item's table entry is loaded
    // then and used at the end, when the last chunk has already fetched the next item's first
    // chunk.  With no more items than CTAs nothing is drawn.
    struct Item {
        int32_t i, j, r0, c_begin, c_end, seq_start, seq_end;
    };
    // One sequence: its offsets must be [0, single_T] (an input, read before grid_dep_wait);
    // otherwise it is taken as empty and only its state passes through.
    const bool single_ok = single_T < 0 || gdn::offsets_single_ok(cu[0], cu[1], single_T);
    const auto decode = [&](int32_t q) {
        Item it;
        const int32_t rank = q / (8 * h_v), rem = q - rank * 8 * h_v;
        it.j = rem >> 3;
        it.r0 = (rem & 7) * kRows;
        if (single_T >= 0) {   // one sequence: chunks 0 .. ceil(T / 64) - 1 of tokens 0 .. T - 1
            it.i = 0;
            it.c_begin = 0;
            it.c_end = single_ok ? (single_T + kC - 1) / kC : 0;
            it.seq_start = 0;
            it.seq_end = single_ok ? single_T : 0;
        } else {               // two independent loads (their use can come much later)
            it.i = order[rank];
            const int4 si = seqinfo[rank];
            it.c_begin = si.x;
            it.c_end = si.y;
            it.seq_start = si.z;
            it.seq_end = si.w;
        }
        return it;
    };

    // phase-2 ownership: key columns c = 16 (warp % 8) + gq (+8), rows r = 8 (warp / 8) + 2 tg (+1)
    const int mc = warp & 7, nr = warp >> 3;
    float st[4] = {0.f, 0.f, 0.f, 0.f};
    // state pieces -> shared memory [r][c] (stmatrix .trans of the [c][r] fragments)
    const uint32_t st_addr = sp_s + sw256(8 * nr + lr, 16 * mc + 8 * (lb & 1));
    const auto store_state = [&]() {
        const Pieces3 lo = split3(st[0], st[1]);   // rows c, pairs (r, r + 1)
        const Pieces3 hi = split3(st[2], st[3]);   // rows c + 8
#pragma unroll
        for (int p = 0; p < 3; ++p) stsm_x2_trans(st_addr + p * kRows * 256, lo.p[p], hi.p[p]);
    };
    // phase-1 / output ownership: tokens m0 .. m0 + 15, state rows n0 .. n0 + 7, key half kh
    const int mt = warp & 3, m0 = 16 * mt, n0 = 8 * ((warp >> 2) & 1), kh = warp >> 3;
    float* mypart = part + (warp & 7) * 128 + lane;   // 4 values x 32 lanes per warp pair
    // causal output steps kk = 0 .. mt: the lower warp takes kk < kmid, the upper the rest
    const int kmid = (mt + 2) >> 1;
    const int kk_lo = kh ? kmid : 0, kk_hi = kh ? mt + 1 : kmid;

    uint32_t n = 0;            // chunk loads consumed by this CTA: stage n % 2, phase n / 2
    bool have_first = false;   // the current item's first chunk was loaded by the previous item
    const int32_t G = static_cast<int32_t>(gridDim.x);
    const bool draws = kMulti && n_items > G;
    // This kernel may start while the prepare kernel before it still runs.  Until
    // grid_dep_wait() it reads only the call's inputs (the first item's initial state); the
    // chunk list's tables, the workspace and the counter wait for it.
    grid_dep_launch();
    if (single_T < 0) grid_dep_wait();   // order and seqinfo, for the first item
    Item it = decode(blockIdx.x);
    if (tid == 0 && it.c_begin < it.c_end) {   // (this CTA loads chunks: the maps are real)
        gf16::prefetch_tensormap(&map_w);
        gf16::prefetch_tensormap(&map_a);
        gf16::prefetch_tensormap(&map_q);
        gf16::prefetch_tensormap(&map_k);
    }
    for (int32_t q = blockIdx.x; q < n_items;) {
        int32_t qn = n_items;   // the next item, known from the first chunk's middle barrier
        Item nx{};
        const int32_t j = it.j, r0 = it.r0, jq = j / qgroup, jk = j / kgroup;
        const int32_t c_begin = it.c_begin, c_end = it.c_end;
        const int32_t seq_start = it.seq_start, seq_end = it.seq_end;
        const auto chunk_t0 = [&](int32_t ch) { return seq_start + (ch - c_begin) * kC; };
        const auto cj_of = [&](int32_t ch) { return static_cast<int64_t>(ch) * h_v + j; };
        const int64_t sbase = ((static_cast<int64_t>(it.i) * h_v + j) * kD + r0) * kD;
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const int c = 16 * mc + gq + 8 * (e >> 1), r = 8 * nr + 2 * tg + (e & 1);
            st[e] = s0 ? s0[sbase + r * kD + c] : 0.f;
        }
        store_state();
        if (q == static_cast<int32_t>(blockIdx.x)) grid_dep_wait();
        uint32_t drawn = 0;   // (thread 0) the draw for the next item
        if (tid == 0 && draws) drawn = atomicAdd(counter, 1u);
        __syncthreads();   // barriers initialised, state pieces visible
        if (kMulti && c_begin >= c_end) {   // an empty sequence: only its state passes through
            if (tid == 0) *next_item = draws ? G + static_cast<int32_t>(drawn) : n_items;
            __syncthreads();
            qn = *next_item;
            if (qn < n_items) nx = decode(qn);
            __syncthreads();   // all have read next_item
        }
        if (c_begin < c_end && !have_first) {
            if (tid == 0)
                scan_issue(base, n & 1, bar0 + 8 * (n & 1), &map_w, &map_a, &map_q, &map_k, ut,
                           gam, cj_of(c_begin), r0, chunk_t0(c_begin), jq, jk);
            const bool ok = gf16::mbar_wait(bar0 + 8 * (n & 1), (n >> 1) & 1, nullptr, wait_ns);
            if (__syncthreads_or(!ok)) {
                if (tid == 0) atomicOr(status, gdn::kStatusTimeout);
                return;
            }
        }
        float pend[4] = {0.f, 0.f, 0.f, 0.f};   // upper warps: own output partial, stored next chunk
        int32_t pend_t0 = 0, pend_len = 0;
        // upper warps: o = scale (own partial + the lower warp's partial in shared memory)
        const auto flush_output = [&]() {
            const int t = m0 + gq, r = n0 + 2 * tg;
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int tt = t + 8 * h;
                if (tt < pend_len)
                    *reinterpret_cast<uint32_t*>(
                        o + ((static_cast<int64_t>(pend_t0) + tt) * o_tok + j * o_hmul) * kD +
                            r0 + r) =
                        pack_bf16(scale * (pend[2 * h] + mypart[(2 * h) * 32]),
                                  scale * (pend[2 * h + 1] + mypart[(2 * h + 1) * 32]));
            }
            pend_len = 0;
        };

        for (int32_t ch = c_begin; ch < c_end; ++ch) {
            const int b = n & 1;
            const int32_t t0 = chunk_t0(ch);
            const int32_t len = min(kC, seq_end - t0);
            if (kh && pend_len > 0) flush_output();   // before this warp reuses its partial slot
            // the next chunk of this item, or the next item's first chunk (fault == 1, a testing
            // hook: an item's second chunk is never loaded, so the wait for it runs out with nothing
            // in flight)
            if (tid == 0 && ch + 1 < c_end && !(fault == 1 && ch == c_begin))
                scan_issue(base, b ^ 1, bar0 + 8 * (b ^ 1), &map_w, &map_a, &map_q, &map_k, ut,
                           gam, cj_of(ch + 1), r0, chunk_t0(ch + 1), jq, jk);
            const uint32_t sb = base + b * kStageBytes;
            const uint32_t w_s = sb + kOffW, q_s = sb + kOffQ, k_s = sb + kOffK, a_s = sb + kOffA;
            const float* Bup = upf + b * kRows * kC;   // U'^T rows [r][t]
            const float* Bg = gf + b * 2 * kC;         // g_t, then g_C / g_t

            // ---- phase 1: U = U' - W S^T, P = Q S^T over this warp's 64 key columns ----
            float u_hi[4] = {0.f, 0.f, 0.f, 0.f}, u_lo[4] = {0.f, 0.f, 0.f, 0.f},
                  u_l2[4] = {0.f, 0.f, 0.f, 0.f}, pq[4] = {0.f, 0.f, 0.f, 0.f},
                  pq2[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int k4 = 0; k4 < 4; ++k4) {
                const int kk = 4 * kh + k4;
                // A fragments (rows m0 + (lane % 16), columns 16 kk + 8 (lane / 16))
                const int arow = m0 + (lane & 15), acol = 16 * kk + 8 * (lane >> 4);
                uint32_t w0[4], w1[4], w2[4], qa[4];
                ldsm_x4(w0, w_s + tsw(arow, acol, 3 * kC));
                ldsm_x4(w1, w_s + tsw(kC + arow, acol, 3 * kC));
                ldsm_x4(w2, w_s + tsw(2 * kC + arow, acol, 3 * kC));
                ldsm_x4(qa, q_s + tsw(arow, acol, kC));
                // B fragments of the state pieces (rows n0 + lr, columns 16 kk + 8 (lb & 1));
                // x4 blocks 0, 1 = piece 0, blocks 2, 3 = piece 1; x2 = piece 2
                const uint32_t boff = sw256(n0 + lr, 16 * kk + 8 * (lb & 1));
                uint32_t s01[4], s2[2];
                ldsm_x4(s01, sp_s + (lb >> 1) * kRows * 256 + boff);
                ldsm_x2(s2, sp_s + 2 * kRows * 256 + boff);
                mma_bf16(u_hi, w0, s01[0], s01[1]);
                mma_bf16(u_lo, w0, s01[2], s01[3]);
                mma_bf16(u_l2, w1, s01[0], s01[1]);
                mma_bf16(pq, qa, s01[0], s01[1]);
                mma_bf16(u_lo, w0, s2[0], s2[1]);
                mma_bf16(u_l2, w1, s01[2], s01[3]);
                mma_bf16(pq2, qa, s01[2], s01[3]);
                mma_bf16(u_lo, w2, s01[0], s01[1]);
                mma_bf16(pq2, qa, s2[0], s2[1]);
            }
            float u[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                u[e] = u_hi[e] + (u_lo[e] + u_l2[e]);
                pq[e] += pq2[e];
            }
            // (lower warps) the epilogue's U' rows and decay ratios, read before the barrier; the
            // upper warps skip these loads (lanes of one token share a bank: 4-way conflicts)
            const int te = m0 + gq, re = n0 + 2 * tg;
            float f0 = 0.f, f1 = 0.f, up0 = 0.f, up1 = 0.f, up2 = 0.f, up3 = 0.f;
            if (!kh) {
                f0 = Bg[kC + te];
                f1 = Bg[kC + te + 8];
                up0 = Bup[re * kC + te];
                up1 = Bup[(re + 1) * kC + te];
                up2 = Bup[re * kC + te + 8];
                up3 = Bup[(re + 1) * kC + te + 8];
            }
            if (kh) {
#pragma unroll
                for (int e = 0; e < 4; ++e) mypart[e * 32] = u[e];
            }
            if (kMulti && tid == 0 && ch == c_begin)
                *next_item = draws ? G + static_cast<int32_t>(drawn) : n_items;
            __syncthreads();   // upper-half partial U ready (and, at the first chunk, the next item)
            if (kMulti && ch == c_begin) {
                qn = *next_item;
                if (qn < n_items) nx = decode(qn);   // used at the item's end
            }
            if (!kh) {
#pragma unroll
                for (int e = 0; e < 4; ++e) u[e] += mypart[e * 32];
                // U~ = (g_C / g_t)(U' - W S^T) -> pieces [r][t] (stmatrix .trans of [t][r] fragments)
                const float x0 = f0 * (up0 - u[0]);
                const float x1 = f0 * (up1 - u[1]);
                const float x2 = f1 * (up2 - u[2]);
                const float x3 = f1 * (up3 - u[3]);
                const Pieces3 lo = split3(x0, x1), hi = split3(x2, x3);
                // block lb (lanes 8 lb ..): stored row r = n0 + lr, columns t = m0 + 8 lb
                const uint32_t addr = sw128(n0 + lr, m0 + 8 * (lb & 1));
#pragma unroll
                for (int p = 0; p < 3; ++p) stsm_x2_trans(up_s + p * kRows * 128 + addr, lo.p[p], hi.p[p]);
            }
            __syncthreads();   // U~ complete
            // the last chunk: the next item's first chunk goes into the other stage now
            if (kMulti && tid == 0 && ch + 1 == c_end && qn < n_items && nx.c_begin < nx.c_end)
                scan_issue(base, b ^ 1, bar0 + 8 * (b ^ 1), &map_w, &map_a, &map_q, &map_k, ut, gam,
                           static_cast<int64_t>(nx.c_begin) * h_v + nx.j, nx.r0, nx.seq_start,
                           nx.j / qgroup, nx.j / kgroup);

            // ---- phase 2a: S_next^T[c][r] = g_C S^T + K^T U~ over tokens t (4 steps of 16) ----
            {
                const float gc = Bg[kC - 1];
                float acc[4] = {gc * st[0], gc * st[1], gc * st[2], gc * st[3]};
                float acc2[4] = {0.f, 0.f, 0.f, 0.f}, acc3[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                for (int kk = 0; kk < kC / 16; ++kk) {
                    // A = K^T: ldmatrix .trans of k rows t = 16 kk + lr + 8 (lane / 16), columns
                    // c = 16 mc + 8 ((lane / 8) % 2)
                    uint32_t ka[4];
                    ldsm_x4_trans(ka, k_s + tsw(16 * kk + lr + 8 * (lane >> 4), 16 * mc + 8 * (lb & 1), kC));
                    // B = U~ pieces [r][t], rows 8 nr + lr: x4 = pieces 0, 1; x2 = piece 2
                    const uint32_t boff = sw128(8 * nr + lr, 16 * kk + 8 * (lb & 1));
                    uint32_t u01[4], u2[2];
                    ldsm_x4(u01, up_s + (lb >> 1) * kRows * 128 + boff);
                    ldsm_x2(u2, up_s + 2 * kRows * 128 + boff);
                    mma_bf16(acc, ka, u01[0], u01[1]);
                    mma_bf16(acc2, ka, u01[2], u01[3]);
                    mma_bf16(acc3, ka, u2[0], u2[1]);
                }
#pragma unroll
                for (int e = 0; e < 4; ++e) st[e] = acc[e] + (acc2[e] + acc3[e]);
            }

            // ---- phase 2b: this warp's share of O = diag(g) P + A' U~ (tokens s <= t) ----
            {
                const int t = m0 + gq;
                float oacc[4] = {Bg[t] * pq[0], Bg[t] * pq[1], Bg[t + 8] * pq[2], Bg[t + 8] * pq[3]};
                for (int kk = kk_lo; kk < kk_hi; ++kk) {
                    const int arow = m0 + (lane & 15), acol = 16 * kk + 8 * (lane >> 4);
                    uint32_t a0[4], a1[4];
                    ldsm_x4(a0, a_s + sw128(arow, acol));
                    ldsm_x4(a1, a_s + sw128(kC + arow, acol));
                    // U~ pieces 0 and 1, rows n0 + lr: blocks 0, 1 = piece 0, 2, 3 = piece 1
                    uint32_t ub[4];
                    ldsm_x4(ub, up_s + (lb >> 1) * kRows * 128 + sw128(n0 + lr, 16 * kk + 8 * (lb & 1)));
                    mma_bf16(oacc, a0, ub[0], ub[1]);
                    mma_bf16(oacc, a0, ub[2], ub[3]);
                    mma_bf16(oacc, a1, ub[0], ub[1]);
                }
                if (!kh) {
#pragma unroll
                    for (int e = 0; e < 4; ++e) mypart[e * 32] = oacc[e];
                } else {
#pragma unroll
                    for (int e = 0; e < 4; ++e) pend[e] = oacc[e];
                    pend_t0 = t0;
                    pend_len = len;
                }
            }
            store_state();
            {
                const bool more =
                    ch + 1 < c_end || (kMulti && qn < n_items && nx.c_begin < nx.c_end);
                const bool ok = !more || gf16::mbar_wait(bar0 + 8 * (b ^ 1), ((n + 1) >> 1) & 1,
                                                         nullptr, wait_ns);
                if (__syncthreads_or(!ok)) {   // state pieces complete, the next chunk landed
                    if (tid == 0) atomicOr(status, gdn::kStatusTimeout);
                    return;
                }
            }
            ++n;
        }
        if (kh && pend_len > 0) flush_output();
        if (s_final)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int c = 16 * mc + gq + 8 * (e >> 1), r = 8 * nr + 2 * tg + (e & 1);
                s_final[sbase + r * kD + c] = st[e];
            }
        have_first = c_begin < c_end && qn < n_items && nx.c_begin < nx.c_end;
        q = qn;
        it = nx;
    }
}

// ---- the same scan with its chunk products on the fifth-generation tensor cores -------------------
// One CTA per work item (sequence, value head, block of 16 state rows), as gdn_scan_kernel; the
// chunk's operands arrive by TMA into the same double-buffered stages (the q rows beside the W
// pieces, see below).  Every product is one tcgen05.mma stream issued by one thread, reading its
// operands from shared memory and accumulating in tensor memory, with the fp32 pieces stacked
// along M and N so that each shared-memory tile is read once per product:
//   P1   D_a = [W0; W1] [S0; S1; S2]^T      (M 128: tokens of pieces 0 and 1; N 48; K 128)
//        D_b = [W2; Q ] [S0; S1; S2]^T      (M 128: tokens of piece 2 and of q)
//        U   = W0 (S0 + S1 + S2) + W1 (S0 + S1) + W2 S0     (the six terms of order <= 2)
//        P   = Q (S0 + S1 + S2)
//   P2   D_2 = K^T [U~0; U~1; U~2]^T        (M 128: key columns; N 48; K 64 tokens; K^T read
//                                           MN-major straight from the q/k tile)
//        S_next = g_C S + (the three column blocks of D_2)
//   P3   D_3 = [A'0; A'1] [U~0; U~1]^T      (M 128; N 32; K 64)
//        O   = scale (g P + A'0 (U~0 + U~1) + A'1 U~0)
// Precision as in gdn_scan_kernel (three bfloat16 pieces per fp32 operand, the terms of order
// <= 2), with the pieces cut by truncation, which makes x0 + x1 + x2 = x exact.
// The state S (fp32, 16 rows x 128 columns) lives in registers: thread (lane quarter lq, half h)
// holds rows 8h .. 8h + 7 of column 32 lq + lane; its three bfloat16 pieces are written to shared
// memory in the K-major layout P1 reads.  Every epilogue is spread over all eight warps.  P3
// commits to its own barrier and a chunk's outputs are finished while the next chunk's P1 runs,
// so only P1 -> U~ -> P2 -> S sits on the chain from chunk to chunk.
namespace tc {
constexpr int kThreads = 256;

// Layout of the scan for kR state rows per CTA (16 or 32).  Offsets in bytes from a
// 1024-byte-aligned base; every operand tile 1024-byte aligned.
//   stage s (two of them): per 64-column half h of the 128 key columns, at s * kStage + h * 32 KB,
//     the rows W0 (64), W1 (64), W2 (64), q (64), 128-byte swizzle; with kR = 16 also the k tile
//     (two 64-column halves of 64 token rows) and the A' pieces (128 rows of 64 tokens)
//   with kR = 32 the k tile and the A' pieces are single-buffered after the stages, loaded a
//   chunk ahead as soon as the previous chunk's P2 and P3 have read them (shared memory has no
//   room for a second copy beside the wider state and U~ pieces)
//   U'^T rows [stage][kR][64] f32, the decays [stage][g_t | g_C / g_t] f32, the state pieces,
//   the U~ pieces, the exchange buffer [kR][64] f32, the barriers, the TMEM address, the next item
template <int kR>
struct Cfg {
    static constexpr bool kSingleKA = kR == 32;
    static constexpr int kRH = kR / 2;                 // state rows per thread
    static constexpr uint32_t kN1 = 3 * kR;            // N of P1 and P2 (three pieces)
    static constexpr uint32_t kN3 = 2 * kR;            // N of P3 (two pieces)
    static constexpr uint32_t kHalf = 32768;
    static constexpr uint32_t kOffW2 = 16384;          // [W2; q] inside a half
    static constexpr uint32_t kOffQ = 24576;
    static constexpr uint32_t kStage = kSingleKA ? 65536 : 98304;
    static constexpr uint32_t kOffK = kSingleKA ? 2 * kStage : 65536;            // in-stage for 16
    static constexpr uint32_t kOffA = kSingleKA ? 2 * kStage + 16384 : 81920;
    static constexpr uint32_t kOffUp = kSingleKA ? 2 * kStage + 32768 : 2 * kStage;
    static constexpr uint32_t kUpBytes = kR * kC * 4;
    static constexpr uint32_t kOffG = kOffUp + 2 * kUpBytes;
    static constexpr uint32_t kSbo = 128;                       // between core matrices along N
    static constexpr uint32_t kLbo = (kN1 / 8) * 128;           // between core matrices along K
    static constexpr uint32_t kOffB1 = kOffG + 2 * 2 * kC * 4;  // state pieces: kN1 x 128 bf16
    static constexpr uint32_t kOffB2 = kOffB1 + 16 * kLbo;      // U~ pieces: kN1 x 64 bf16
    static constexpr uint32_t kOffX = kOffB2 + 8 * kLbo;        // exchange [kR][64] f32
    static constexpr uint32_t kOffBar = kOffX + kR * kC * 4;    // barriers (7 slots)
    static constexpr uint32_t kOffSlot = kOffBar + 7 * 8;
    static constexpr uint32_t kOffItem = kOffSlot + 4;
    static constexpr size_t kSmem = kOffItem + 4 + 1024;
    // bytes the stage barrier counts per chunk
    static constexpr uint32_t kStageTx =
        2 * (3 * kC * 128 + kC * 128) + (kSingleKA ? 0 : 2 * (2 * kC * 128)) + kUpBytes + 2 * kC * 4;
    // tensor-memory columns: D_a, D_b, D_2 (kN1 each), D_3 (kN3)
    static constexpr uint32_t kColA = 0, kColB = kN1, kCol2 = 2 * kN1, kCol3 = 3 * kN1;
    static constexpr uint32_t kCols = kR == 16 ? 256 : 512;
    static_assert(kOffB1 % 1024 == 0 && kOffB2 % 1024 == 0, "operand tiles");
    static_assert(kSmem <= 232448, "tcgen05 scan shared memory");
    static_assert(kCol3 + kN3 <= kCols, "tensor-memory columns");
};

// The state pieces (B of P1: N = 3 kR rows n = kR p + r, K = 128 key columns) and the U~ pieces
// (B of P2 and P3: N = 3 kR or 2 kR, K = 64 tokens) are MN-major tiles without swizzle: 8 x 8
// core matrices of 128 contiguous bytes (8 K rows of 8 consecutive n), kSbo = 128 bytes apart
// along N and kLbo = 3 kR / 8 x 128 bytes apart along K.  A thread holding 8 consecutive rows n
// of one K index writes them as one 16-byte store.
template <int kR>
__device__ __forceinline__ uint32_t piece_off(int n, int k)
{
    return static_cast<uint32_t>((n >> 3) * Cfg<kR>::kSbo + (k >> 3) * Cfg<kR>::kLbo +
                                 (k & 7) * 16 + (n & 7) * 2);
}
// Shared-memory descriptor of such a tile (no swizzle: layout field 0).
template <int kR>
__device__ __forceinline__ uint64_t desc_mn_none(uint32_t smem_addr)
{
    uint64_t d = 0;
    d |= static_cast<uint64_t>((smem_addr & 0x3FFFFu) >> 4);
    d |= static_cast<uint64_t>((Cfg<kR>::kLbo >> 4) & 0x3FFFu) << 16;
    d |= static_cast<uint64_t>((Cfg<kR>::kSbo >> 4) & 0x3FFFu) << 32;
    d |= static_cast<uint64_t>(1u) << 46;
    return d;
}
// Pieces of 8 values as three 16-byte rows of bfloat16 (value e in element e).  The split is by
// truncation: x0 keeps the sign, exponent and top 7 mantissa bits of x (the low 16 bits of its
// fp32 pattern cleared), x - x0 is exact in fp32, x1 is its truncation the same way and
// x2 = x - x0 - x1 has at most 8 significant bits, so x0 + x1 + x2 = x exactly (for normal
// values whose pieces stay normal) with |x1| < 2^-7 |x| and |x2| < 2^-15 |x|.  The high halves
// of two fp32 patterns make one bfloat16x2 word (byte permute).
__device__ __forceinline__ void store_pieces8(uint32_t addr0, uint32_t piece_stride,
                                              const float* v)
{
    uint32_t w[3][4];
#pragma unroll
    for (int e = 0; e < 8; e += 2) {
        uint32_t p[2][3];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const float x = v[e + h];
            const uint32_t x0 = __float_as_uint(x) & 0xFFFF0000u;
            const float r1 = x - __uint_as_float(x0);
            const uint32_t x1 = __float_as_uint(r1) & 0xFFFF0000u;
            const float r2 = r1 - __uint_as_float(x1);
            p[h][0] = x0;
            p[h][1] = x1;
            p[h][2] = __float_as_uint(r2);
        }
#pragma unroll
        for (int pc = 0; pc < 3; ++pc) w[pc][e / 2] = __byte_perm(p[0][pc], p[1][pc], 0x7632);
    }
#pragma unroll
    for (int pc = 0; pc < 3; ++pc)
        gf16::st_shared_v4(addr0 + pc * piece_stride, w[pc][0], w[pc][1], w[pc][2], w[pc][3]);
}
// 8 consecutive 32-bit columns of the thread's own TMEM lane.
__device__ __forceinline__ void tmem_ld8(uint32_t taddr, uint32_t* r)
{
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]),
                   "=r"(r[6]), "=r"(r[7])
                 : "r"(taddr));
}
// n consecutive columns (a multiple of 8) of the thread's own TMEM lane.
template <int n>
__device__ __forceinline__ void tmem_ldn(uint32_t taddr, uint32_t (&r)[n])
{
#pragma unroll
    for (int i = 0; i < n; i += 8) tmem_ld8(taddr + i, r + i);
}
// Shared-memory descriptor of an MN-major operand with the 128-byte swizzle: 64 MN elements per
// 128-byte row, 8 K rows per 1024-byte atom (SBO between atoms along K), atoms along MN LBO apart.
__device__ __forceinline__ uint64_t desc_mn_sw128(uint32_t smem_addr, uint32_t lbo, uint32_t sbo)
{
    uint64_t d = 0;
    d |= static_cast<uint64_t>((smem_addr & 0x3FFFFu) >> 4);
    d |= static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16;
    d |= static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32;
    d |= static_cast<uint64_t>(1u) << 46;
    d |= static_cast<uint64_t>(2u) << 61;
    return d;
}

// One thread: announce a chunk's stage bytes on the stage barrier and start those loads (W, q,
// the block's U'^T rows and the decays; with kR = 16 also k and A').
template <int kR>
__device__ __forceinline__ void issue(uint32_t base, int s, uint32_t bar, const CUtensorMap* map_w,
                                      const CUtensorMap* map_a, const CUtensorMap* map_q,
                                      const CUtensorMap* map_k, const float* __restrict__ ut,
                                      const float* __restrict__ gam, int64_t cj, int32_t r0,
                                      int32_t t0, int32_t jq, int32_t jk)
{
    using C = Cfg<kR>;
    gf16::mbar_arrive_expect_tx(bar, C::kStageTx);
    const uint32_t st = base + s * C::kStage;
    const int32_t yw = static_cast<int32_t>(cj * 3 * kC);
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        gf16::tma_load_2d(st + h * C::kHalf, map_w, bar, 64 * h, yw);            // W0, W1, W2
        gf16::tma_load_3d(st + h * C::kHalf + C::kOffQ, map_q, bar, 64 * h, jq, t0);
        if constexpr (!C::kSingleKA)
            gf16::tma_load_3d(st + C::kOffK + h * kC * 128, map_k, bar, 64 * h, jk, t0);
    }
    if constexpr (!C::kSingleKA)
        gf16::tma_load_2d(st + C::kOffA, map_a, bar, 0, static_cast<int32_t>(cj * 2 * kC));
    bulk_g2s(base + C::kOffUp + s * C::kUpBytes, ut + (cj * kD + r0) * kC, C::kUpBytes, bar);
    bulk_g2s(base + C::kOffG + s * 2 * kC * 4, gam + cj * 2 * kC, 2 * kC * 4, bar);
}
// kR = 32: the single-buffered k tile of a chunk (tokens t0 .., key head jk) on `bar`.
__device__ __forceinline__ void issue_k(uint32_t dst, uint32_t bar, const CUtensorMap* map_k,
                                        int32_t t0, int32_t jk)
{
    gf16::mbar_arrive_expect_tx(bar, 2 * kC * 128);
#pragma unroll
    for (int h = 0; h < 2; ++h) gf16::tma_load_3d(dst + h * kC * 128, map_k, bar, 64 * h, jk, t0);
}
// kR = 32: the single-buffered A' pieces of chunk cj on `bar`.
__device__ __forceinline__ void issue_a(uint32_t dst, uint32_t bar, const CUtensorMap* map_a,
                                        int64_t cj)
{
    gf16::mbar_arrive_expect_tx(bar, 2 * kC * 128);
    gf16::tma_load_2d(dst, map_a, bar, 0, static_cast<int32_t>(cj * 2 * kC));
}
}  // namespace tc

template <bool kMulti, int kR>
__global__ void __launch_bounds__(tc::kThreads, 1)
    gdn_scan_tc_kernel(const __grid_constant__ CUtensorMap map_w,
                       const __grid_constant__ CUtensorMap map_a,
                       const __grid_constant__ CUtensorMap map_q,
                       const __grid_constant__ CUtensorMap map_k, const int32_t* __restrict__ order,
                       const int4* __restrict__ seqinfo, uint32_t* __restrict__ counter,
                       int32_t n_items, const float* __restrict__ ut,
                       const float* __restrict__ gam, const float* __restrict__ s0,
                       float* __restrict__ s_final, __nv_bfloat16* __restrict__ o,
                       uint32_t* __restrict__ status, int32_t h_v, int32_t qgroup, int32_t kgroup,
                       int32_t o_tok, int32_t o_hmul, float scale,
                       uint64_t wait_ns, uint32_t fault, int32_t single_T,
                       const int32_t* __restrict__ cu)
{
    using C = tc::Cfg<kR>;
    constexpr int RH = C::kRH;                 // state rows per thread
    constexpr int kBlocks = kD / kR;           // row blocks per head
    extern __shared__ __align__(16) uint8_t smraw[];
    const uint32_t raw = smem_u32(smraw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t* gbase = smraw + (base - raw);
    const float* upf = reinterpret_cast<const float*>(gbase + C::kOffUp);
    const float* gf = reinterpret_cast<const float*>(gbase + C::kOffG);
    float* xch = reinterpret_cast<float*>(gbase + C::kOffX);   // [kR rows][64 tokens]
    volatile int32_t* next_item = reinterpret_cast<volatile int32_t*>(gbase + C::kOffItem);
    const uint32_t b1_s = base + C::kOffB1, b2_s = base + C::kOffB2;
    // barriers: stage 0, stage 1, P1, P2, P3, and (kR = 32) the k tile and the A' pieces
    const uint32_t bar_full = base + C::kOffBar, bar_p1 = bar_full + 16, bar_p2 = bar_full + 24,
                   bar_p3 = bar_full + 32, bar_k = bar_full + 40, bar_a = bar_full + 48;
    const int tid = threadIdx.x, warp = tid / 32, lane = tid % 32;
    // Thread roles.  Tensor-memory lane quarter lq = warp % 4 holds rows 32 lq .. + 31 of every
    // accumulator; the two warps of a quarter split the kR state rows, rh = RH (warp / 4) ...
    //   quarters 0-1: the W0 / W2 rows of P1, i.e. token t = 32 lq + lane: U, then U~
    //   quarters 2-3: the W1 / q rows, token t = 32 (lq - 2) + lane: the W1 partial of U, P, O
    //   every quarter in P2: key column c = 32 lq + lane: the state S[rh .. rh + RH - 1][c]
    const int lq = warp & 3, rh = RH * (warp >> 2);
    const int t_lo = 32 * lq + lane;          // token of quarters 0-1
    const int t_hi = 32 * (lq - 2) + lane;    // token of quarters 2-3
    const int c_me = 32 * lq + lane;          // key column in P2

    if (tid == 0) {
#pragma unroll
        for (int i = 0; i < 7; ++i) gf16::mbar_init(bar_full + 8 * i, 1);
        gf16::fence_mbarrier_init();
    }
    if (warp == 0) {
        gf16::tmem_alloc<1>(base + C::kOffSlot, C::kCols);
        gf16::tmem_relinquish<1>();
    }

    // Work items as in gdn_scan_kernel, with kBlocks row blocks of kR rows per head: item q ->
    // rank q / (kBlocks h_v), head (q / kBlocks) % h_v, rows kR (q % kBlocks) ...; CTA b starts
    // with item b and draws each later one from `counter`.
    struct Item {
        int32_t i, j, r0, c_begin, c_end, seq_start, seq_end;
    };
    const bool single_ok = single_T < 0 || gdn::offsets_single_ok(cu[0], cu[1], single_T);
    const auto decode = [&](int32_t q) {
        Item it;
        const int32_t rank = q / (kBlocks * h_v), rem = q - rank * kBlocks * h_v;
        it.j = rem / kBlocks;
        it.r0 = (rem % kBlocks) * kR;
        if (single_T >= 0) {
            it.i = 0;
            it.c_begin = 0;
            it.c_end = single_ok ? (single_T + kC - 1) / kC : 0;
            it.seq_start = 0;
            it.seq_end = single_ok ? single_T : 0;
        } else {
            it.i = order[rank];
            const int4 si = seqinfo[rank];
            it.c_begin = si.x;
            it.c_end = si.y;
            it.seq_start = si.z;
            it.seq_end = si.w;
        }
        return it;
    };

    // instruction descriptors: bf16 x bf16 -> f32, M 128; every B is MN-major (bit 16), P2's A
    // (K^T from the k tile) too (bit 15)
    const uint32_t id1 = gf16::make_idesc_f16(128, C::kN1, 1) | (1u << 16);
    const uint32_t id3 = gf16::make_idesc_f16(128, C::kN3, 1) | (1u << 16);
    const uint32_t id1_mn = id1 | (1u << 15);
    const uint64_t d_b1 = tc::desc_mn_none<kR>(b1_s);
    const uint64_t d_b2 = tc::desc_mn_none<kR>(b2_s);
    constexpr uint32_t kStepB = (2 * C::kLbo) >> 4;   // a K step of 16: two core matrices

    const int32_t G = static_cast<int32_t>(gridDim.x);
    const bool draws = kMulti && n_items > G;
    grid_dep_launch();
    if (single_T < 0) grid_dep_wait();   // order and seqinfo, for the first item
    Item it = decode(blockIdx.x);
    if (tid == 0 && it.c_begin < it.c_end) {
        gf16::prefetch_tensormap(&map_w);
        gf16::prefetch_tensormap(&map_a);
        gf16::prefetch_tensormap(&map_q);
        gf16::prefetch_tensormap(&map_k);
    }
    gf16::tcgen05_fence_before();
    __syncthreads();
    gf16::tcgen05_fence_after();
    const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(gbase + C::kOffSlot);
    const uint32_t tl = tmem + (static_cast<uint32_t>(32 * lq) << 16);   // this quarter's lanes

    // S[rh + e][c_me], e < RH: this thread's part of the state, fp32, chunk to chunk
    float S[RH];
    const auto store_state = [&]() {
#pragma unroll
        for (int e = 0; e < RH; e += 8)
            tc::store_pieces8(b1_s + tc::piece_off<kR>(rh + e, c_me), (kR / 8) * C::kSbo, S + e);
        gf16::fence_proxy_async_smem();
    };
    // Outputs of a chunk are finished during the next chunk's P1 (or after an item's last
    // chunk): quarters 2-3 keep their P = Q S^T rows and the decays g_t until then.
    float P[RH];
    float pend_g = 0.f;
    int32_t pend_t0 = 0, pend_len = 0, pend_j = 0, pend_r0 = 0;
    bool pend = false;
    uint32_t pend_par = 0;
    bool failed = false;
    // kR = 32: loads of the single-buffered k / A' tiles issued and not yet consumed (their
    // barriers complete once per chunk, in order, so the parity of the next completion is the
    // number of completions so far, mod 2)
    uint32_t k_issued = 0, a_issued = 0, k_done = 0, a_done = 0;
    const auto issue_k = [&](int32_t t0_, int32_t jk_) {
        if (tid == 128) tc::issue_k(base + C::kOffK, bar_k, &map_k, t0_, jk_);
        __syncwarp();
        ++k_issued;
    };
    const auto issue_a = [&](int64_t cj_) {
        if (tid == 128) tc::issue_a(base + C::kOffA, bar_a, &map_a, cj_);
        __syncwarp();
        ++a_issued;
    };
    // O = scale (g P + A'0 (U~0 + U~1) + A'1 U~0) of the pending chunk: quarters 0-1 pass the
    // A'0 sums through xch; quarters 2-3 add their A'1 U~0 and write o.
    const auto flush_output = [&]() {
        failed |= !gf16::mbar_wait(bar_p3, pend_par, nullptr, wait_ns);
        gf16::tcgen05_fence_after();
        uint32_t x[RH], y[RH];
        if (lq < 2) {
            tc::tmem_ldn<RH>(tl + C::kCol3 + rh, x);
            tc::tmem_ldn<RH>(tl + C::kCol3 + kR + rh, y);
            gf16::tmem_ld_wait();
#pragma unroll
            for (int e = 0; e < RH; ++e)
                xch[(rh + e) * kC + t_lo] = __uint_as_float(x[e]) + __uint_as_float(y[e]);
        } else {
            tc::tmem_ldn<RH>(tl + C::kCol3 + rh, x);
            gf16::tmem_ld_wait();
        }
        gf16::tcgen05_fence_before();
        __syncthreads();
        if (lq >= 2 && t_hi < pend_len) {
            __nv_bfloat16* dst = o + ((static_cast<int64_t>(pend_t0) + t_hi) * o_tok +
                                      pend_j * o_hmul) * kD + pend_r0 + rh;
#pragma unroll
            for (int e0 = 0; e0 < RH; e0 += 8) {
                uint32_t w[4];
#pragma unroll
                for (int e = e0; e < e0 + 8; e += 2)
                    w[(e - e0) / 2] = pack_bf16(
                        scale * fmaf(pend_g, P[e], __uint_as_float(x[e]) + xch[(rh + e) * kC + t_hi]),
                        scale * fmaf(pend_g, P[e + 1],
                                     __uint_as_float(x[e + 1]) + xch[(rh + e + 1) * kC + t_hi]));
                *reinterpret_cast<uint4*>(dst + e0) = make_uint4(w[0], w[1], w[2], w[3]);
            }
        }
        pend = false;
        if constexpr (C::kSingleKA) __syncthreads();   // xch is written again in epilogue 1
    };

    uint32_t n = 0;            // chunks this CTA consumed: stage n % 2, barrier phases
    bool have_first = false;
    for (int32_t q = blockIdx.x; q < n_items;) {
        int32_t qn = n_items;
        Item nx{};
        const int32_t j = it.j, r0 = it.r0, jq = j / qgroup, jk = j / kgroup;
        const int32_t c_begin = it.c_begin, c_end = it.c_end;
        const int32_t seq_start = it.seq_start, seq_end = it.seq_end;
        const auto chunk_t0 = [&](int32_t ch) { return seq_start + (ch - c_begin) * kC; };
        const auto cj_of = [&](int32_t ch) { return static_cast<int64_t>(ch) * h_v + j; };
        const int64_t sbase = ((static_cast<int64_t>(it.i) * h_v + j) * kD + r0) * kD;
#pragma unroll
        for (int e = 0; e < RH; ++e) S[e] = s0 ? s0[sbase + (rh + e) * kD + c_me] : 0.f;
        store_state();
        if (q == static_cast<int32_t>(blockIdx.x)) grid_dep_wait();
        uint32_t drawn = 0;
        if (tid == 0 && draws) drawn = atomicAdd(counter, 1u);
        __syncthreads();   // state pieces visible
        if (kMulti && c_begin >= c_end) {   // an empty sequence: only its state passes through
            if (tid == 0) *next_item = draws ? G + static_cast<int32_t>(drawn) : n_items;
            __syncthreads();
            qn = *next_item;
            if (qn < n_items) nx = decode(qn);
            __syncthreads();
        }
        if (c_begin < c_end && !have_first) {
            if (tid == 0)
                tc::issue<kR>(base, n & 1, bar_full + 8 * (n & 1), &map_w, &map_a, &map_q, &map_k,
                              ut, gam, cj_of(c_begin), r0, chunk_t0(c_begin), jq, jk);
            if constexpr (C::kSingleKA) {
                issue_k(chunk_t0(c_begin), jk);
                issue_a(cj_of(c_begin));
            }
            const bool ok =
                gf16::mbar_wait(bar_full + 8 * (n & 1), (n >> 1) & 1, nullptr, wait_ns);
            if (__syncthreads_or(!ok)) {
                if (tid == 0) atomicOr(status, gdn::kStatusTimeout);
                failed = true;
                break;
            }
        }

        for (int32_t ch = c_begin; ch < c_end; ++ch) {
            const int b = n & 1;
            const uint32_t par = n & 1;   // phase parity of the MMA barriers (and k, A')
            const int32_t t0 = chunk_t0(ch);
            const int32_t len = min(kC, seq_end - t0);
            const bool next_in_item = ch + 1 < c_end && !(fault == 1 && ch == c_begin);
            // (warp 4 issues the loads, so that warp 0 goes straight to the MMAs).  With kR = 16
            // the other stage still holds the previous chunk's A' pieces, which its output
            // product P3 may still be reading: the loads wait for that product first.
            if (next_in_item) {
                if constexpr (!C::kSingleKA) {
                    if (tid == 128 && pend)
                        failed |= !gf16::mbar_wait(bar_p3, pend_par, nullptr, wait_ns);
                }
                if (tid == 128)
                    tc::issue<kR>(base, b ^ 1, bar_full + 8 * (b ^ 1), &map_w, &map_a, &map_q,
                                  &map_k, ut, gam, cj_of(ch + 1), r0, chunk_t0(ch + 1), jq, jk);
                __syncwarp();   // warp 4 whole again before any .aligned instruction
            }
            const uint32_t sb = base + b * C::kStage;
            const float* Bup = upf + b * (C::kUpBytes / 4);
            const float* Bg = gf + b * 2 * kC;
            const uint32_t k_tile = C::kSingleKA ? base + C::kOffK : sb + C::kOffK;
            const uint32_t a_tile = C::kSingleKA ? base + C::kOffA : sb + C::kOffA;

            // ---- P1: D_a = [W0; W1] [S0; S1; S2]^T, D_b = [W2; q] [S0; S1; S2]^T ----
            if (warp == 0) {
                if (gf16::elect_one_sync()) {
                    gf16::tcgen05_fence_after();
                    const uint64_t d_st = gf16::make_smem_desc_sw128(sb, 1024);
#pragma unroll
                    for (int kk = 0; kk < 8; ++kk) {
                        const uint32_t ka = ((kk >> 2) * C::kHalf + (kk & 3) * 32) >> 4;
                        const uint32_t kb = kk * kStepB;
                        gf16::mma_f16<1>(tmem + C::kColA, d_st + ka, d_b1 + kb, id1, kk > 0);
                        gf16::mma_f16<1>(tmem + C::kColB, d_st + ka + (C::kOffW2 >> 4),
                                         d_b1 + kb, id1, kk > 0);
                    }
                    gf16::mma_commit(bar_p1);
                }
                __syncwarp();
            }
            // the previous chunk's outputs, while P1 runs; after them (kR = 32) this chunk's A'
            // pieces may replace the previous chunk's
            if (pend) {
                flush_output();
                if constexpr (C::kSingleKA) {
                    if (ch != c_begin) issue_a(cj_of(ch));
                }
            }

            // ---- epilogue 1 ----
            float u[8];
            failed |= !gf16::mbar_wait(bar_p1, par, nullptr, wait_ns);
            gf16::tcgen05_fence_after();
            if constexpr (kR == 16) {
                // U partial (quarters 0-1): W0 (S0 + S1 + S2) + W2 S0; quarters 2-3 pass
                // W1 (S0 + S1) through xch and keep P = q (S0 + S1 + S2) for the outputs
                if (lq < 2) {
                    uint32_t x[8], y[8], z[8], w[8];
                    tc::tmem_ld8(tl + C::kColA + rh, x);
                    tc::tmem_ld8(tl + C::kColA + kR + rh, y);
                    tc::tmem_ld8(tl + C::kColA + 2 * kR + rh, z);
                    tc::tmem_ld8(tl + C::kColB + rh, w);
                    gf16::tmem_ld_wait();
#pragma unroll
                    for (int e = 0; e < 8; ++e)
                        u[e] = (__uint_as_float(x[e]) + __uint_as_float(y[e])) +
                               (__uint_as_float(z[e]) + __uint_as_float(w[e]));
                } else {
                    uint32_t x[8], y[8], z[8], w[8], v[8];
                    tc::tmem_ld8(tl + C::kColA + rh, x);
                    tc::tmem_ld8(tl + C::kColA + kR + rh, y);
                    tc::tmem_ld8(tl + C::kColB + rh, z);
                    tc::tmem_ld8(tl + C::kColB + kR + rh, w);
                    tc::tmem_ld8(tl + C::kColB + 2 * kR + rh, v);
                    gf16::tmem_ld_wait();
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        xch[(rh + e) * kC + t_hi] = __uint_as_float(x[e]) + __uint_as_float(y[e]);
                        P[e] = __uint_as_float(z[e]) +
                               (__uint_as_float(w[e]) + __uint_as_float(v[e]));
                    }
                    pend_g = Bg[t_hi];
                }
            } else {
                // 16 rows per thread: quarters 0-1 keep the U partial of rows rh .. rh + 7 and
                // pass rows rh + 8 .. to quarters 2-3, which pass their W1 partial of rows
                // rh .. rh + 7 back; each side then finishes 8 rows of its token
                if (lq < 2) {
                    uint32_t x[16], y[16], z[16], w[16];
                    tc::tmem_ldn<16>(tl + C::kColA + rh, x);
                    tc::tmem_ldn<16>(tl + C::kColA + kR + rh, y);
                    tc::tmem_ldn<16>(tl + C::kColA + 2 * kR + rh, z);
                    tc::tmem_ldn<16>(tl + C::kColB + rh, w);
                    gf16::tmem_ld_wait();
#pragma unroll
                    for (int e = 0; e < 16; ++e) {
                        const float v = (__uint_as_float(x[e]) + __uint_as_float(y[e])) +
                                        (__uint_as_float(z[e]) + __uint_as_float(w[e]));
                        if (e < 8) u[e] = v;
                        else xch[(rh + e) * kC + t_lo] = v;
                    }
                } else {
                    uint32_t x[16], y[16];
                    tc::tmem_ldn<16>(tl + C::kColA + rh, x);
                    tc::tmem_ldn<16>(tl + C::kColA + kR + rh, y);
                    gf16::tmem_ld_wait();
#pragma unroll
                    for (int e = 0; e < 16; ++e) {
                        const float w1 = __uint_as_float(x[e]) + __uint_as_float(y[e]);
                        if (e < 8) xch[(rh + e) * kC + t_hi] = w1;
                        else u[e - 8] = w1;
                    }
                    tc::tmem_ldn<16>(tl + C::kColB + rh, x);
                    tc::tmem_ldn<16>(tl + C::kColB + kR + rh, y);
                    gf16::tmem_ld_wait();
#pragma unroll
                    for (int e = 0; e < 16; ++e) P[e] = __uint_as_float(x[e]) + __uint_as_float(y[e]);
                    tc::tmem_ldn<16>(tl + C::kColB + 2 * kR + rh, x);
                    gf16::tmem_ld_wait();
#pragma unroll
                    for (int e = 0; e < 16; ++e) P[e] += __uint_as_float(x[e]);
                    pend_g = Bg[t_hi];
                }
            }
            if (kMulti && tid == 0 && ch == c_begin)
                *next_item = draws ? G + static_cast<int32_t>(drawn) : n_items;
            gf16::tcgen05_fence_before();
            if (__syncthreads_or(failed)) {   // partials exchanged (and the next item)
                // an MMA wait ran out: report, let the loads in flight land, stop
                failed = true;
                if (tid == 0) atomicOr(status, gdn::kStatusTimeout);
                if (tid == 128 && next_in_item)
                    gf16::mbar_wait(bar_full + 8 * (b ^ 1), ((n + 1) >> 1) & 1, nullptr, wait_ns);
                break;
            }
            if (kMulti && ch == c_begin) {
                qn = *next_item;
                if (qn < n_items) nx = decode(qn);
            }
            // U~ = (g_C / g_t)(U' - U) -> pieces [kR p + r][t]; every load first: the stores
            // below are ordered asm statements
            if constexpr (kR == 16) {
                if (lq < 2) {
                    const float f = Bg[kC + t_lo];
                    float v[8];
#pragma unroll
                    for (int e = 0; e < 8; ++e)
                        v[e] = f * (Bup[(rh + e) * kC + t_lo] - (u[e] + xch[(rh + e) * kC + t_lo]));
                    tc::store_pieces8(b2_s + tc::piece_off<kR>(rh, t_lo), (kR / 8) * C::kSbo, v);
                    gf16::fence_proxy_async_smem();
                }
            } else {
                const int t = lq < 2 ? t_lo : t_hi;
                const int r8 = lq < 2 ? rh : rh + 8;
                const float f = Bg[kC + t];
                float v[8];
#pragma unroll
                for (int e = 0; e < 8; ++e)
                    v[e] = f * (Bup[(r8 + e) * kC + t] - (u[e] + xch[(r8 + e) * kC + t]));
                tc::store_pieces8(b2_s + tc::piece_off<kR>(r8, t), (kR / 8) * C::kSbo, v);
                gf16::fence_proxy_async_smem();
            }
            __syncthreads();   // U~ pieces complete; the exchange buffer is free again
            // ---- P2 (state) ----
            bool k_ok = true;
            if (warp == 0) {
                if constexpr (C::kSingleKA) {   // this chunk's k tile has landed
                    k_ok = gf16::mbar_wait(bar_k, k_done & 1, nullptr, wait_ns);
                }
                if (gf16::elect_one_sync() && k_ok) {
                    gf16::tcgen05_fence_after();
                    const uint64_t d_k = tc::desc_mn_sw128(k_tile, kC * 128, 1024);
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk)
                        gf16::mma_f16<1>(tmem + C::kCol2, d_k + ((kk * 2048) >> 4),
                                         d_b2 + kk * kStepB, id1_mn, kk > 0);
                    gf16::mma_commit(bar_p2);
                }
                __syncwarp();
            }
            if constexpr (C::kSingleKA) ++k_done;
            failed |= !k_ok;
            // the last chunk: the next item's first chunk goes into the other stage now
            const bool next_item_first =
                kMulti && ch + 1 == c_end && qn < n_items && nx.c_begin < nx.c_end;
            if (next_item_first) {
                if (tid == 128)
                    tc::issue<kR>(base, b ^ 1, bar_full + 8 * (b ^ 1), &map_w, &map_a, &map_q,
                                  &map_k, ut, gam, static_cast<int64_t>(nx.c_begin) * h_v + nx.j,
                                  nx.r0, nx.seq_start, nx.j / qgroup, nx.j / kgroup);
                __syncwarp();
            }
            {   // ---- epilogue 2: S_next = g_C S + K^T U~ ----
                failed |= !(k_ok && gf16::mbar_wait(bar_p2, par, nullptr, wait_ns));
                gf16::tcgen05_fence_after();
                // P3 (outputs) behind P2 in the tensor pipe: issued by warp 4 once P2 is done
                // (and, kR = 32, once this chunk's A' pieces have landed), so warp 0 goes on
                // to its part of the state at once
                if (warp == 4) {
                    bool a_ok = true;
                    if constexpr (C::kSingleKA)
                        a_ok = gf16::mbar_wait(bar_a, a_done & 1, nullptr, wait_ns);
                    if (gf16::elect_one_sync() && a_ok) {
                        const uint64_t d_a = gf16::make_smem_desc_sw128(a_tile, 1024);
#pragma unroll
                        for (int kk = 0; kk < 4; ++kk)
                            gf16::mma_f16<1>(tmem + C::kCol3, d_a + ((kk * 32) >> 4),
                                             d_b2 + kk * kStepB, id3, kk > 0);
                        gf16::mma_commit(bar_p3);
                    }
                    __syncwarp();
                    failed |= !a_ok;
                }
                if constexpr (C::kSingleKA) {
                    ++a_done;
                    // the k tile is free: the next chunk's (of this item, or the next item's
                    // first) comes in now
                    if (next_in_item) issue_k(chunk_t0(ch + 1), jk);
                    else if (next_item_first) issue_k(nx.seq_start, nx.j / kgroup);
                }
                uint32_t x[RH], y[RH], z[RH];
                tc::tmem_ldn<RH>(tl + C::kCol2 + rh, x);
                tc::tmem_ldn<RH>(tl + C::kCol2 + kR + rh, y);
                tc::tmem_ldn<RH>(tl + C::kCol2 + 2 * kR + rh, z);
                gf16::tmem_ld_wait();
                const float gc = Bg[kC - 1];
#pragma unroll
                for (int e = 0; e < RH; ++e)
                    S[e] = fmaf(gc, S[e], __uint_as_float(x[e]) +
                                              (__uint_as_float(y[e]) + __uint_as_float(z[e])));
                store_state();
            }
            pend = true;
            pend_par = par;
            pend_t0 = t0;
            pend_len = len;
            pend_j = j;
            pend_r0 = r0;
            gf16::tcgen05_fence_before();
            {   // state pieces complete, the next chunk landed
                const bool more = ch + 1 < c_end || next_item_first;
                const bool ok = !more || gf16::mbar_wait(bar_full + 8 * (b ^ 1),
                                                         ((n + 1) >> 1) & 1, nullptr, wait_ns);
                failed |= !ok;
                if (__syncthreads_or(failed)) {
                    failed = true;
                    if (tid == 0) atomicOr(status, gdn::kStatusTimeout);
                    break;
                }
            }
            ++n;
        }
        if (failed) break;
        // the item's last outputs (the next item may have no chunk whose P1 they could follow)
        if (pend) {
            flush_output();
            if constexpr (C::kSingleKA) {   // the next item's first A' pieces may come in now
                if (kMulti && qn < n_items && nx.c_begin < nx.c_end)
                    issue_a(static_cast<int64_t>(nx.c_begin) * h_v + nx.j);
            }
            if (__syncthreads_or(failed)) {
                failed = true;
                if (tid == 0) atomicOr(status, gdn::kStatusTimeout);
                break;
            }
        }
        if (s_final)
#pragma unroll
            for (int e = 0; e < RH; ++e) s_final[sbase + (rh + e) * kD + c_me] = S[e];
        have_first = c_begin < c_end && qn < n_items && nx.c_begin < nx.c_end;
        q = qn;
        it = nx;
    }
    // Every MMA this CTA issued has completed before its tensor memory is freed: each commit was
    // waited on, except, after a timeout, that of a chunk's output product, waited on here.  The
    // TMA loads in flight after a timeout are those of one stage at most, which the wait that ran
    // out or the drain above covered, and (kR = 32) k and A' tiles issued but not consumed,
    // waited on here.
    if (tid == 0 && pend) gf16::mbar_wait(bar_p3, pend_par, nullptr, wait_ns);
    if (tid == 128) {
        if (k_issued > k_done) gf16::mbar_wait(bar_k, k_done & 1, nullptr, wait_ns);
        if (a_issued > a_done) gf16::mbar_wait(bar_a, a_done & 1, nullptr, wait_ns);
    }
    gf16::tcgen05_fence_before();
    __syncthreads();
    if (warp == 0) {
        gf16::tcgen05_fence_after();
        gf16::tmem_dealloc<1>(tmem, C::kCols);
    }
}

bool misaligned(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) != 0; }

// Output heads of the head layout (h_q, h_k, h_v), or -1: h_v a multiple of h_k, and either
// h_q == h_k (one output per value head: MHA, GVA) or h_q a multiple of h_v (one output per
// query head, query head m reading state m / (h_q / h_v): GQA).
int64_t out_heads(int64_t h_q, int64_t h_k, int64_t h_v)
{
    if (h_q <= 0 || h_k <= 0 || h_v <= 0 || h_v % h_k != 0) return -1;
    if (h_q == h_k) return h_v;
    if (h_q % h_v == 0) return h_q;
    return -1;
}

int check(const void* q, const void* k, const void* v, const float* alpha, const float* beta,
          const int32_t* cu, int64_t n_seqs, int64_t T, int64_t h_q, int64_t h_k, int64_t h_v,
          int64_t head_dim, const void* o)
{
    if (n_seqs < 0 || T < 0 || h_q <= 0 || h_k <= 0 || h_v <= 0)
        return gdn_fail(GDN_ERR_INVALID_ARG, "negative size or no heads (n_seqs=%lld T=%lld "
                        "h_q=%lld h_k=%lld h_v=%lld)", (long long)n_seqs, (long long)T,
                        (long long)h_q, (long long)h_k, (long long)h_v);
    if (out_heads(h_q, h_k, h_v) < 0)
        return gdn_fail(GDN_ERR_INVALID_ARG, "heads q=%lld k=%lld v=%lld: h_v must be a multiple "
                        "of h_k, and h_q equal h_k or be a multiple of h_v", (long long)h_q,
                        (long long)h_k, (long long)h_v);
    if (head_dim != kD)
        return gdn_fail(GDN_ERR_UNSUPPORTED, "head_dim=%lld; only head_dim 128 is supported",
                        (long long)head_dim);
    if (T > (1ll << 30) || n_seqs > (1ll << 30) || h_v > 65535 || h_q > 65535)
        return gdn_fail(GDN_ERR_INVALID_ARG, "size out of range");
    if (n_seqs == 0) return GDN_OK;
    if (cu == nullptr) return gdn_fail(GDN_ERR_INVALID_ARG, "cu_seqlens is null");
    if (T > 0 && (!q || !k || !v || !alpha || !beta || !o))
        return gdn_fail(GDN_ERR_INVALID_ARG, "a tensor pointer is null");
    if (T > 0 && (misaligned(q) || misaligned(k) || misaligned(v) || misaligned(o)))
        return gdn_fail(GDN_ERR_UNSUPPORTED, "q, k, v and o must be 16-byte aligned");
    return GDN_OK;
}


// ---- TMA descriptors of the scan's operands -----------------------------------------------------
PFN_cuTensorMapEncodeTiled_v12000 gdn_encode_fn()
{
    static PFN_cuTensorMapEncodeTiled_v12000 fn = [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult res{};
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &res) != cudaSuccess ||
            res != cudaDriverEntryPointSuccess)
            p = nullptr;
        return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    }();
    return fn;
}

// A tensor of `rank` dimensions (dims[0] contiguous; strides in bytes of dims 1..), moved in
// boxes of `box` elements with the 128-byte swizzle (box[0] elements = 128 bytes): bfloat16, or
// fp32 when `f32`.
int gdn_make_map(CUtensorMap* map, const void* ptr, uint32_t rank, const cuuint64_t* dims,
                 const cuuint64_t* strides, const cuuint32_t* box, const char* what,
                 bool f32 = false)
{
    auto fn = gdn_encode_fn();
    if (!fn) return gdn_fail(GDN_ERR_CUDA, "cuTensorMapEncodeTiled is not available");
    const cuuint32_t estr[3] = {1, 1, 1};
    const CUresult r = fn(map, f32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
                          rank, const_cast<void*>(ptr), dims,
                          strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                          CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS)
        return gdn_fail(GDN_ERR_CUDA, "cuTensorMapEncodeTiled failed (CUresult %d) for %s", (int)r,
                        what);
    return GDN_OK;
}

// Once per device, under a lock (calls may come from several threads): the device must be an
// sm_103 part, and the kernels' dynamic shared memory above the 48 KB default is raised (an
// attribute of each device's copy of the kernel).
int gdn_ensure_smem(int dev)
{
    static std::mutex mu;
    static bool done[kMaxDevices] = {};
    if (dev < 0 || dev >= kMaxDevices)
        return gdn_fail(GDN_ERR_UNSUPPORTED, "device ordinal %d above %d", dev, kMaxDevices - 1);
    std::lock_guard<std::mutex> lock(mu);
    if (done[dev]) return GDN_OK;
    int major = 0, minor = 0;
    cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
    cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
    if (major != 10 || minor != 3)
        return gdn_fail(GDN_ERR_UNSUPPORTED,
                        "device %d is sm_%d%d; these kernels are built for sm_103a only", dev,
                        major, minor);
    cudaError_t e = cudaFuncSetAttribute(gdn_prepare_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(kPrepSpreadSmem));
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(gdn_scan_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(kScanSmem));
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(gdn_scan_kernel<false>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(kScanSmem));
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(gdn_scan_tc_kernel<true, 16>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(tc::Cfg<16>::kSmem));
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(gdn_scan_tc_kernel<false, 16>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(tc::Cfg<16>::kSmem));
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(gdn_scan_tc_kernel<true, 32>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(tc::Cfg<32>::kSmem));
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(gdn_scan_tc_kernel<false, 32>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(tc::Cfg<32>::kSmem));
    if (e != cudaSuccess)
        return gdn_fail(GDN_ERR_CUDA, "cudaFuncSetAttribute (dynamic shared memory): %s",
                        cudaGetErrorString(e));
    done[dev] = true;
    return GDN_OK;
}

// Launches `kernel` on `stream` with programmatic stream serialization: it may start as soon as
// every CTA of the kernel before it has called grid_dep_launch() (or at once, when that kernel
// never does), and waits in grid_dep_wait() for it to finish before it touches what that kernel
// may write.  A call's first kernel waits before it touches any memory at all (the kernel before
// it belongs to the caller), so consecutive calls, and a call after a GEMM of this library,
// overlap their launch gaps.
// GDN_PDL=0 (read once per process) launches a call's first kernel the plain way instead, for
// comparison; its wait then returns at once.
bool gdn_first_pdl()
{
    static const bool v = [] {
        const char* e = std::getenv("GDN_PDL");
        return !(e && e[0] == '0');
    }();
    return v;
}
// GDN_PREP_SPREAD=0 (read once per process) keeps the prepare kernel's two-CTAs-per-SM shared
// memory size for grids of at most one CTA per SM too, for comparison.
bool gdn_prep_spread()
{
    static const bool v = [] {
        const char* e = std::getenv("GDN_PREP_SPREAD");
        return !(e && e[0] == '0');
    }();
    return v;
}

template <typename... KArgs, typename... Args>
cudaError_t gdn_launch(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t stream, bool first, Args... args)
{
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = (first && !gdn_first_pdl()) ? 0u : 1u;
    return cudaLaunchKernelEx(&cfg, kernel, args...);
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

int gdn_prefill_heads(const void* q, const void* k, const void* v, const float* alpha,
                      const float* beta, const int32_t* cu_seqlens, int64_t n_seqs,
                      int64_t total_tokens, int64_t h_q, int64_t h_k, int64_t h_v,
                      int64_t head_dim, float scale, const float* initial_state, void* o,
                      float* final_state, void* workspace, size_t workspace_bytes,
                      cudaStream_t stream)
{
    t_gdn_error.clear();
    int rc = check(q, k, v, alpha, beta, cu_seqlens, n_seqs, total_tokens, h_q, h_k, h_v,
                   head_dim, o);
    if (rc != GDN_OK || n_seqs == 0) return rc;
    const WsLayout l = layout_for(total_tokens, n_seqs, h_v);
    if (workspace == nullptr || workspace_bytes < l.total || misaligned(workspace))
        return gdn_fail(GDN_ERR_INVALID_ARG, "workspace of %zu bytes (16-byte aligned) needed",
                        l.total);
    auto* ws = static_cast<uint8_t*>(workspace);
    auto* status = reinterpret_cast<uint32_t*>(ws + l.status);
    auto* order = reinterpret_cast<int32_t*>(ws + l.order);
    auto* counter = reinterpret_cast<uint32_t*>(ws + l.counter);
    auto* seqinfo = reinterpret_cast<int4*>(ws + l.seqinfo);
    auto* chunk_offset = reinterpret_cast<int32_t*>(ws + l.chunk_offset);
    auto* n_chunks = reinterpret_cast<int32_t*>(ws + l.n_chunks);
    auto* chunks = reinterpret_cast<int4*>(ws + l.chunks);
    auto* wp = reinterpret_cast<__nv_bfloat16*>(ws + l.wp);
    auto* ap = reinterpret_cast<__nv_bfloat16*>(ws + l.ap);
    auto* ut = reinterpret_cast<float*>(ws + l.ut);
    auto* gm = reinterpret_cast<float*>(ws + l.gam);
    const int64_t mc = max_chunks_for(total_tokens, n_seqs);
    if (n_seqs * h_v * (kD / kRows) >= (int64_t(1) << 31))
        return gdn_fail(GDN_ERR_UNSUPPORTED, "too many sequences x value heads for one call");
    if (mc * h_v * 3 * kC >= (int64_t(1) << 31))
        return gdn_fail(GDN_ERR_UNSUPPORTED, "too many chunks x value heads for one call (%lld)",
                        (long long)(mc * h_v));

    // Heads.  State head j reads key head j / kgroup.  With h_q == h_k its one output is output
    // head j and its query head j / kgroup (one pass).  With grouped queries (h_q a multiple of
    // h_v) it serves query heads j r + g, g < r = h_q / h_v, written to output heads j r + g:
    // pass g runs the whole pipeline on the strided view of q that holds heads j r + g (the state
    // recurrence does not read q, so every pass reproduces the same states; only the last pass
    // writes the final states).
    const int64_t h_o = out_heads(h_q, h_k, h_v);
    const int64_t passes = h_o == h_v ? 1 : h_q / h_v;
    const int32_t kgroup = static_cast<int32_t>(h_v / h_k);
    const int32_t qgroup = passes == 1 ? kgroup : 1;

    // One sequence with tokens: cu_seqlens is [0, total_tokens] by contract, so the kernels
    // number the chunks themselves and the chunk-list launch is skipped.
    const int32_t single_T = (n_seqs == 1 && total_tokens > 0) ? static_cast<int32_t>(total_tokens)
                                                                : -1;
    const int64_t n_items = n_seqs * h_v * (kD / kRows);
    const int scan_kernel = g_gdn_scan.load();
    int dev = 0, sms = 0;
    cudaError_t e = cudaSuccess;
    if ((e = cudaGetDevice(&dev)) != cudaSuccess ||
        (e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
        return gdn_fail(GDN_ERR_CUDA, "device query: %s", cudaGetErrorString(e));
    if ((rc = gdn_ensure_smem(dev)) != GDN_OK) return rc;

    // TMA descriptors that do not depend on the pass: W pieces [cj * 192 rows][128] (stored by
    // the prepare kernel, loaded by the scan), U'^T [cj * 128 rows][64] fp32 (stored), A' pieces
    // [cj * 128 rows][64], k as {128, h_k, total_tokens}, v as {128, h_v, total_tokens}.  With no
    // tokens nothing is moved and they stay zero.
    CUtensorMap map_w{}, map_ut{}, map_a{}, map_k{}, map_v{};
    const cuuint32_t bq[3] = {64, 1, kC};
    if (total_tokens > 0) {
        const cuuint64_t dw[2] = {static_cast<cuuint64_t>(kD), static_cast<cuuint64_t>(mc * h_v * 3 * kC)};
        const cuuint64_t sw[1] = {kD * 2};
        const cuuint32_t bw[2] = {64, 3 * kC};
        const cuuint64_t du[2] = {static_cast<cuuint64_t>(kC), static_cast<cuuint64_t>(mc * h_v * kD)};
        const cuuint64_t su[1] = {kC * 4};
        const cuuint32_t bu[2] = {32, kD};
        const cuuint64_t da[2] = {static_cast<cuuint64_t>(kC), static_cast<cuuint64_t>(mc * h_v * 2 * kC)};
        const cuuint64_t sa[1] = {kC * 2};
        const cuuint32_t ba[2] = {64, 2 * kC};
        const cuuint64_t dk3[3] = {static_cast<cuuint64_t>(kD), static_cast<cuuint64_t>(h_k),
                                   static_cast<cuuint64_t>(total_tokens)};
        const cuuint64_t sk3[2] = {kD * 2, static_cast<cuuint64_t>(h_k) * kD * 2};
        const cuuint64_t dv3[3] = {static_cast<cuuint64_t>(kD), static_cast<cuuint64_t>(h_v),
                                   static_cast<cuuint64_t>(total_tokens)};
        const cuuint64_t sv3[2] = {kD * 2, static_cast<cuuint64_t>(h_v) * kD * 2};
        if ((rc = gdn_make_map(&map_w, wp, 2, dw, sw, bw, "W pieces")) != GDN_OK ||
            (rc = gdn_make_map(&map_ut, ut, 2, du, su, bu, "U'^T", true)) != GDN_OK ||
            (rc = gdn_make_map(&map_a, ap, 2, da, sa, ba, "A' pieces")) != GDN_OK ||
            (rc = gdn_make_map(&map_k, k, 3, dk3, sk3, bq, "k")) != GDN_OK ||
            (rc = gdn_make_map(&map_v, v, 3, dv3, sv3, bq, "v")) != GDN_OK)
            return rc;
    }
    // q as seen by pass g: h_q heads (one pass), or the h_v heads j r + g (stride r heads)
    CUtensorMap map_q[8];
    const int64_t map_passes = total_tokens > 0 ? passes : 1;
    if (map_passes > 8)
        return gdn_fail(GDN_ERR_UNSUPPORTED, "more than 8 query heads per state head");
    for (int64_t gp = 0; gp < map_passes; ++gp) {
        map_q[gp] = CUtensorMap{};
        if (total_tokens == 0) continue;
        const cuuint64_t dq[3] = {static_cast<cuuint64_t>(kD),
                                  static_cast<cuuint64_t>(passes == 1 ? h_q : h_v),
                                  static_cast<cuuint64_t>(total_tokens)};
        const cuuint64_t sq[2] = {static_cast<cuuint64_t>(passes) * kD * 2,
                                  static_cast<cuuint64_t>(h_q) * kD * 2};
        if ((rc = gdn_make_map(&map_q[gp], static_cast<const __nv_bfloat16*>(q) + gp * kD, 3, dq,
                               sq, bq, "q")) != GDN_OK)
            return rc;
    }

    // Each kernel may start while the one before it finishes (programmatic dependent launch:
    // the kernels wait for their predecessor before they touch what it writes, and the call's
    // first kernel, the chunk list or the first pass's prepare, before it touches anything).
    if (single_T < 0) {
        e = gdn_launch(gdn_chunk_list_kernel, dim3(1), dim3(1024), 0, stream, true, cu_seqlens,
                       static_cast<int32_t>(n_seqs), static_cast<int32_t>(total_tokens),
                       chunk_offset, chunks,
                       static_cast<int32_t>(mc), n_chunks, status, order, seqinfo, counter);
        if (e != cudaSuccess)
            return gdn_fail(GDN_ERR_CUDA, "gdn_chunk_list_kernel: %s", cudaGetErrorString(e));
    }
    // with no tokens every state only passes through: one pass.  Every pass reads the initial
    // states and the last one writes the final states, so the two may be one buffer.
    for (int64_t gp = 0; gp < map_passes; ++gp) {
        if (mc > 0 && total_tokens > 0) {
            // two CTAs fit on an SM; a grid with no more CTAs than SMs takes one per SM, which
            // measured 7% faster per call on 1024 tokens x 8 heads (128 CTAs)
            const dim3 pgrid(static_cast<uint32_t>(mc), static_cast<uint32_t>(h_v));
            const size_t psmem =
                gdn_prep_spread() && mc * h_v <= sms ? kPrepSpreadSmem : kPrepSmem;
            e = gdn_launch(gdn_prepare_kernel, pgrid, dim3(kPrepThreads), psmem, stream,
                           single_T >= 0 && gp == 0, map_q[gp], map_k, map_v, map_w, map_ut,
                           alpha, beta,
                           static_cast<const int4*>(chunks), static_cast<const int32_t*>(n_chunks),
                           static_cast<int32_t>(h_v), qgroup, kgroup,
                           static_cast<int32_t>(gp == 0), ap, gm, single_T, cu_seqlens, status,
                           counter, g_gdn_wait_ns.load(),
                           static_cast<int32_t>(single_T >= 0 && gp == 0));
            if (e != cudaSuccess)
                return gdn_fail(GDN_ERR_CUDA, "gdn_prepare_kernel: %s", cudaGetErrorString(e));
        }
        // persistent scan: one CTA per SM (at most one per work item) taking items dynamically;
        // its chunk products on tcgen05 (default) or on mma.sync.  The tcgen05 scan takes 32
        // state rows per item (N 96 per MMA, about the cost of N 48) when 16-row items would
        // give every SM at least eight: it halves the MMAs per row where throughput, not the
        // length of one chain, sets the time.  With fewer items, 16-row items finish sooner and
        // balance better (measured: 20 packed sequences x 16 value heads, 17 items per SM, 260
        // against 325 us; 10 x 8, 4 per SM, 97 against 92 us).
        const bool tensor_core = scan_kernel != GDN_SCAN_MMA_SYNC;
        const bool wide = tensor_core && scan_kernel != GDN_SCAN_TENSOR_CORE_16 &&
                          (scan_kernel == GDN_SCAN_TENSOR_CORE_32 || n_items >= 8 * sms);
        const int64_t items = wide ? n_items / 2 : n_items;
        const int64_t ctas = items < sms ? items : sms;
        auto* scan = !tensor_core ? (items > sms ? gdn_scan_kernel<true> : gdn_scan_kernel<false>)
                     : wide ? (items > sms ? gdn_scan_tc_kernel<true, 32>
                                           : gdn_scan_tc_kernel<false, 32>)
                            : (items > sms ? gdn_scan_tc_kernel<true, 16>
                                           : gdn_scan_tc_kernel<false, 16>);
        e = gdn_launch(scan, dim3(static_cast<uint32_t>(ctas)),
                       dim3(tensor_core ? tc::kThreads : kScanThreads),
                       !tensor_core ? kScanSmem : wide ? tc::Cfg<32>::kSmem : tc::Cfg<16>::kSmem,
                       stream, false, map_w, map_a, map_q[gp], map_k,
                       static_cast<const int32_t*>(single_T >= 0 ? nullptr : order),
                       static_cast<const int4*>(single_T >= 0 ? nullptr : seqinfo), counter,
                       static_cast<int32_t>(items), static_cast<const float*>(ut),
                       static_cast<const float*>(gm), initial_state,
                       gp == map_passes - 1 ? final_state : nullptr,
                       static_cast<__nv_bfloat16*>(o) + gp * kD, status,
                       static_cast<int32_t>(h_v), qgroup, kgroup, static_cast<int32_t>(h_o),
                       static_cast<int32_t>(passes), scale, g_gdn_wait_ns.load(),
                       g_gdn_fault.load(), single_T, cu_seqlens);
        if (e != cudaSuccess)
            return gdn_fail(GDN_ERR_CUDA, "gdn_scan_kernel: %s", cudaGetErrorString(e));
    }
    return GDN_OK;
}

int gdn_prefill(const void* q, const void* k, const void* v, const float* alpha,
                const float* beta, const int32_t* cu_seqlens, int64_t n_seqs,
                int64_t total_tokens, int64_t h_qk, int64_t h_v, int64_t head_dim, float scale,
                const float* initial_state, void* o, float* final_state, void* workspace,
                size_t workspace_bytes, cudaStream_t stream)
{
    return gdn_prefill_heads(q, k, v, alpha, beta, cu_seqlens, n_seqs, total_tokens, h_qk, h_qk,
                             h_v, head_dim, scale, initial_state, o, final_state, workspace,
                             workspace_bytes, stream);
}

const char* gdn_last_error(void) { return t_gdn_error.c_str(); }

int gdn_check_status(const void* workspace, cudaStream_t stream)
{
    t_gdn_error.clear();
    if (workspace == nullptr) return gdn_fail(GDN_ERR_INVALID_ARG, "workspace is null");
    uint32_t word = 0;
    cudaError_t e = cudaMemcpyAsync(&word, static_cast<const uint8_t*>(workspace) +
                                               layout_for(0, 0, 1).status,
                                    sizeof(word), cudaMemcpyDeviceToHost, stream);
    if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
    if (e != cudaSuccess)
        return gdn_fail(GDN_ERR_CUDA, "reading the status word: %s", cudaGetErrorString(e));
    if (word & gdn::kStatusBadOffsets)
        return gdn_fail(GDN_ERR_INVALID_ARG, "cu_seqlens broke its contract (it must start at 0, "
                        "end at total_tokens and never decrease); no token was processed");
    if (word != 0)
        return gdn_fail(GDN_ERR_TIMEOUT, "a scan CTA gave up a bounded wait for its chunk loads");
    return GDN_OK;
}

int gdn_check_offsets(const int32_t* cu_seqlens, int64_t n_seqs, int64_t total_tokens,
                      int64_t h_v, void* workspace, size_t workspace_bytes, cudaStream_t stream)
{
    t_gdn_error.clear();
    if (n_seqs < 0 || total_tokens < 0 || h_v <= 0)
        return gdn_fail(GDN_ERR_INVALID_ARG, "negative size or no heads");
    if (total_tokens > (1ll << 30) || n_seqs > (1ll << 30))
        return gdn_fail(GDN_ERR_INVALID_ARG, "size out of range");
    if (cu_seqlens == nullptr) return gdn_fail(GDN_ERR_INVALID_ARG, "cu_seqlens is null");
    const WsLayout l = layout_for(total_tokens, n_seqs, h_v);
    if (workspace == nullptr || workspace_bytes < l.total || misaligned(workspace))
        return gdn_fail(GDN_ERR_INVALID_ARG, "workspace of %zu bytes (16-byte aligned) needed",
                        l.total);
    auto* ws = static_cast<uint8_t*>(workspace);
    const cudaError_t e = gdn_launch(
        gdn_chunk_list_kernel, dim3(1), dim3(1024), 0, stream, true, cu_seqlens,
        static_cast<int32_t>(n_seqs), static_cast<int32_t>(total_tokens),
        reinterpret_cast<int32_t*>(ws + l.chunk_offset), reinterpret_cast<int4*>(ws + l.chunks),
        static_cast<int32_t>(max_chunks_for(total_tokens, n_seqs)),
        reinterpret_cast<int32_t*>(ws + l.n_chunks), reinterpret_cast<uint32_t*>(ws + l.status),
        reinterpret_cast<int32_t*>(ws + l.order), reinterpret_cast<int4*>(ws + l.seqinfo),
        reinterpret_cast<uint32_t*>(ws + l.counter));
    if (e != cudaSuccess)
        return gdn_fail(GDN_ERR_CUDA, "gdn_chunk_list_kernel: %s", cudaGetErrorString(e));
    return GDN_OK;
}

int gdn_offsets_valid_host(const int32_t* cu_seqlens, int64_t n_seqs, int64_t total_tokens)
{
    if (cu_seqlens == nullptr || n_seqs < 0) return 0;
    for (int64_t i = 0; i < n_seqs; ++i)
        if (!gdn::offsets_pair_ok(cu_seqlens[i], cu_seqlens[i + 1])) return 0;
    return gdn::offsets_ends_ok(cu_seqlens[0], cu_seqlens[n_seqs], total_tokens) ? 1 : 0;
}

int gdn_set_wait_timeout_ms(uint32_t ms)
{
    if (ms == 0) return gdn_fail(GDN_ERR_INVALID_ARG, "timeout must be at least 1 ms");
    g_gdn_wait_ns.store(static_cast<uint64_t>(ms) * 1000000ull);
    return GDN_OK;
}

int gdn_set_scan_kernel(int kernel)
{
    if (kernel < GDN_SCAN_AUTO || kernel > GDN_SCAN_TENSOR_CORE_32)
        return gdn_fail(GDN_ERR_INVALID_ARG, "unknown scan kernel %d", kernel);
    g_gdn_scan.store(kernel);
    return GDN_OK;
}

int gdn_set_fault_injection(int mode)
{
    if (mode < 0 || mode > 1) return gdn_fail(GDN_ERR_INVALID_ARG, "unknown injection %d", mode);
    g_gdn_fault.store(static_cast<uint32_t>(mode));
    return GDN_OK;
}

}  // extern "C"
