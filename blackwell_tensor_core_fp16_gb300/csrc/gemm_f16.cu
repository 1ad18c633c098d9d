// Host side of libgemm_f16.so: argument checks, TMA descriptors, variant choice and launch.
// The C ABI is declared (and documented) in include/gemm_f16.h.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <atomic>
#include <cstdarg>
#include <cstdint>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <string>

#include "../../include/gemm_f16.h"
#include "desc.h"
#include "gemm_kernels.cuh"

namespace {

constexpr int kVersion = 1 * 10000 + 0 * 100 + 0;
constexpr int kMaxDevices = 64;

thread_local std::string t_last_error;

int fail(int code, const char* fmt, ...)
{
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    std::vsnprintf(buf, sizeof(buf), fmt, ap);
    va_end(ap);
    t_last_error = buf;
    return code;
}

int cuda_fail(cudaError_t e, const char* what)
{
    return fail(GEMM_F16_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorString(e), cudaGetErrorName(e));
}

// ---- configuration read once from the environment --------------------------------------------
// Wall-clock limit of one bounded wait inside a kernel: GEMM_F16_WAIT_TIMEOUT_MS at first use
// (default 4000 ms), changeable with gemm_f16_set_wait_timeout_ms.
std::atomic<uint64_t> g_timeout_ns{0};
std::atomic<uint32_t> g_debug_flags{0};

uint64_t wait_timeout_ns()
{
    uint64_t v = g_timeout_ns.load(std::memory_order_relaxed);
    if (v == 0) {
        const char* s = std::getenv("GEMM_F16_WAIT_TIMEOUT_MS");
        long long ms = s ? std::atoll(s) : 4000;
        if (ms < 1) ms = 1;
        v = static_cast<uint64_t>(ms) * 1000000ull;
        uint64_t expected = 0;
        g_timeout_ns.compare_exchange_strong(expected, v);
        v = g_timeout_ns.load(std::memory_order_relaxed);
    }
    return v;
}

uint32_t debug_flags() { return g_debug_flags.load(std::memory_order_relaxed); }

// L2 priorities for the A and B loads and the D stores: bits 1:0 A, bits 3:2 B, bits 5:4 D
// (0 normal, 1 evict_first, 2 evict_last).  Default: A and B evict_last, D normal.  A band of A
// rows is reused by every tile of its group of tile-rows, and a band of B rows by every group
// that sweeps it; with A alone evict_last the runs were 0.5-1.5% faster than with no hint, and
// B evict_last too added 0.5% on 8192^3 and 1.6% on the MLP shape (700-step loops, two
// alternations on one box; B evict_first, B normal and A normal were slower).  D stores with
// evict_first measured within noise (+0.3%), and would push out a result the next kernel often
// reads, so D stays normal.  GEMM_F16_L2_A / GEMM_F16_L2_B / GEMM_F16_L2_D = normal | first |
// last override.
uint32_t l2_hint_setting()
{
    static const uint32_t v = [] {
        auto parse = [](const char* s, uint32_t dflt) -> uint32_t {
            if (!s) return dflt;
            if (!std::strcmp(s, "first")) return 1u;
            if (!std::strcmp(s, "last")) return 2u;
            return 0u;
        };
        return parse(std::getenv("GEMM_F16_L2_A"), 2u) |
               (parse(std::getenv("GEMM_F16_L2_B"), 2u) << 2) |
               (parse(std::getenv("GEMM_F16_L2_D"), 0u) << 4);
    }();
    return v;
}

// Programmatic dependent launch of the GEMM kernels (default on; GEMM_F16_PDL=0 turns it
// off).  With it, a GEMM launched right after another on the same stream does its set-up
// (barriers, tensor memory, descriptor prefetch) on SMs the previous one has left, and only its
// first global-memory access waits for the previous kernel to finish.
bool pdl_setting()
{
    static const bool v = [] {
        const char* s = std::getenv("GEMM_F16_PDL");
        return !(s && s[0] == '0');
    }();
    return v;
}

// Tile-rows per raster group: GEMM_F16_GROUP overrides (1..64); 0 when unset.
uint32_t group_m_override()
{
    static const uint32_t v = [] {
        const char* s = std::getenv("GEMM_F16_GROUP");
        if (!s) return 0u;
        long g = std::atol(s);
        if (g < 1) g = 1;
        if (g > 64) g = 64;
        return static_cast<uint32_t>(g);
    }();
    return v;
}

// Raster group size.  A group of G tile-rows walks the N tiles together, so every B tile is
// loaded once per group instead of once per tile-row, while the group's G row bands of A
// (mma_m rows x K each) stay resident in L2 for the whole sweep.  The rule: the largest power of
// two, at most 16, whose A bands fill no more than a third of L2.  On a GB300 (about 126 MiB of
// L2) with 256-row fp16 tiles this gives 8 at K = 8192 (4 MiB bands) and 16 at K = 4096; a
// sustained sweep of 8, 12, 16 and 20 measured those two as the fastest for 8192^3 and
// 16384x14336x4096 respectively.
uint32_t group_m_for(int64_t mma_m, int64_t K, int64_t elem_bytes, int64_t l2_bytes)
{
    if (const uint32_t o = group_m_override()) return o;
    const int64_t band = mma_m * K * elem_bytes;
    uint32_t g = 1;
    while (g < 16 && band * (2 * g) * 3 <= l2_bytes) g *= 2;
    return g;
}

// ---- the variants ----------------------------------------------------------------------------
using Ws128x256 = gf16::WsCfg<1, 256, 4, true>;
using WsPair = gf16::WsCfg<2, 256, 6, true>;
using Ws128x128 = gf16::WsCfg<1, 128, 6, true>;
using WsPairDirect = gf16::WsCfg<2, 256, 7, false>;
using WsPair192 = gf16::WsCfg<2, 192, 6, true>;

bool variant_info(int v, gemm_f16_variant_info* o)
{
    switch (v) {
    case GEMM_F16_VARIANT_TILE:
        *o = {1, 128, 128, 64, 2, (int)gf16::TileCfg<128>::THREADS,
              (int)gf16::TileCfg<128>::SMEM_ALLOC, (int)gf16::TileCfg<128>::TMEM_COLS,
              (int)gf16::TileCfg<128>::STAGE_TX, 0};
        return true;
    case GEMM_F16_VARIANT_WS_128x256:
        *o = {1, 128, 256, 64, 4, (int)Ws128x256::THREADS, (int)Ws128x256::SMEM_ALLOC,
              (int)Ws128x256::TMEM_COLS, (int)Ws128x256::STAGE_TX, 1};
        return true;
    case GEMM_F16_VARIANT_WS_PAIR:
        *o = {2, 256, 256, 64, 6, (int)WsPair::THREADS, (int)WsPair::SMEM_ALLOC,
              (int)WsPair::TMEM_COLS, (int)WsPair::STAGE_TX, 1};
        return true;
    case GEMM_F16_VARIANT_WS_128x128:
        *o = {1, 128, 128, 64, 6, (int)Ws128x128::THREADS, (int)Ws128x128::SMEM_ALLOC,
              (int)Ws128x128::TMEM_COLS, (int)Ws128x128::STAGE_TX, 1};
        return true;
    case GEMM_F16_VARIANT_WS_PAIR_DIRECT:
        *o = {2, 256, 256, 64, 7, (int)WsPairDirect::THREADS, (int)WsPairDirect::SMEM_ALLOC,
              (int)WsPairDirect::TMEM_COLS, (int)WsPairDirect::STAGE_TX, 1};
        return true;
    case GEMM_F16_VARIANT_WS_PAIR_256x192:
        *o = {2, 256, 192, 64, 6, (int)WsPair192::THREADS, (int)WsPair192::SMEM_ALLOC,
              (int)WsPair192::TMEM_COLS, (int)WsPair192::STAGE_TX, 1};
        return true;
    default:
        return false;
    }
}

int64_t cdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }

// Automatic variant, from bench.py --sweep on GB300 (back-to-back launches): the CTA pair on
// 2048^3, 3000x5000x1000 (34.5 us against 49.9 us for 128x256), 8192^3 and the MLP shape;
// 128x128 tiles where neither larger tile keeps half the SMs busy.
int choose_variant(int64_t M, int64_t N, int64_t K, int num_sms)
{
    if (num_sms < 2) num_sms = 2;
    // A few tiles of short K: the one-tile kernel with its N tile narrowed to spread D over more
    // SMs (128 x 128 x 64: 1.82 us per launch against 2.95 us for the persistent 128 x 128
    // kernel, graph-replayed; 1024 x 1024 x 256: 3.89 against 4.02 us; with K = 512 the
    // persistent kernel's deeper pipeline wins, 4.97 against 5.17 us at 512^3).
    if (K <= 256 && cdiv(M, 128) * cdiv(N, 128) <= num_sms) return GEMM_F16_VARIANT_TILE;
    const int64_t pair_tiles = cdiv(M, 256) * cdiv(N, 256);
    const int64_t tiles_128x256 = cdiv(M, 128) * cdiv(N, 256);
    // The CTA pair once its tiles occupy at least half the SMs: it loads 32 KB per CTA and
    // k-block against 48 KB for a lone 128 x 256 CTA, so a single wave of it is not starved by
    // L2 (2048^3, 64 pair tiles: 14.95 us against 16.8 us for 128 x 256, back-to-back launches
    // with programmatic dependent launch); then 128 x 256 while its tiles fill half the SMs;
    // else 128 x 128.
    if (M > 128 && 4 * pair_tiles >= num_sms) return GEMM_F16_VARIANT_WS_PAIR;
    if (2 * tiles_128x256 >= num_sms) return GEMM_F16_VARIANT_WS_128x256;
    return GEMM_F16_VARIANT_WS_128x128;
}

// ---- per-device state ------------------------------------------------------------------------
// Kernel slots (one per compiled kernel instance) for the per-device caches below:
// 16-bit path: variant + (bf16 ? GEMM_F16_NUM_VARIANTS : 0); block-scaled path: kMxSlot0 +
// 2 * variant + (bf16 output ? 1 : 0); the one-tile kernel's four N tiles: 56 .. 59.
constexpr int kMxSlot0 = 32;
constexpr int kNumSlots = 64;

struct DeviceState {
    bool ready = false;
    int sms = 0;
    int64_t l2_bytes = 0;
    bool smem_set[kNumSlots] = {};    // max dynamic shared memory raised, per kernel slot
    int pair_clusters[kNumSlots] = {};  // co-resident CTA pairs, per kernel slot
};

std::mutex g_mu;
DeviceState g_dev[kMaxDevices];

int device_state(DeviceState** out)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    if (dev < 0 || dev >= kMaxDevices) return fail(GEMM_F16_ERR_CUDA, "device %d out of range", dev);
    std::lock_guard<std::mutex> lk(g_mu);
    DeviceState& d = g_dev[dev];
    if (!d.ready) {
        int major = 0, minor = 0;
        if ((e = cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
            return cuda_fail(e, "cudaDeviceGetAttribute(SM count)");
        int l2 = 0;
        if ((e = cudaDeviceGetAttribute(&l2, cudaDevAttrL2CacheSize, dev)) != cudaSuccess)
            return cuda_fail(e, "cudaDeviceGetAttribute(L2 size)");
        d.l2_bytes = l2;
        cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
        if (major != 10 || minor != 3)
            return fail(GEMM_F16_ERR_UNSUPPORTED,
                        "device %d is sm_%d%d; this library is built for sm_103a only", dev, major,
                        minor);
        d.ready = true;
    }
    *out = &d;
    return GEMM_F16_OK;
}

template <typename Kernel>
int ensure_smem(DeviceState& d, int slot, Kernel kernel, uint32_t bytes)
{
    std::lock_guard<std::mutex> lk(g_mu);
    if (d.smem_set[slot]) return GEMM_F16_OK;
    cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(bytes));
    if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute(max dynamic shared memory)");
    d.smem_set[slot] = true;
    return GEMM_F16_OK;
}

// ---- TMA descriptors -------------------------------------------------------------------------
PFN_cuTensorMapEncodeTiled_v12000 encode_fn()
{
    static PFN_cuTensorMapEncodeTiled_v12000 fn = [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q{};
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) != cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            p = nullptr;
        return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    }();
    return fn;
}

// A row-major matrix of `rows` x `cols` (cols contiguous) of 16-bit elements (fp16, or bf16),
// or of 8-bit codes (fp8: FP8 operands of the block-scaled path), read or written in boxes of
// box_rows x box_cols elements with the 128-byte swizzle (box_cols * element size == 128 bytes).
int make_map(CUtensorMap* map, const void* ptr, uint64_t rows, uint64_t cols, uint32_t box_rows,
             uint32_t box_cols, bool bf16 = false, bool fp8 = false)
{
    auto fn = encode_fn();
    if (!fn) return fail(GEMM_F16_ERR_CUDA, "cuTensorMapEncodeTiled is not available");
    const cuuint64_t dims[2] = {cols, rows};
    const cuuint64_t strides[1] = {cols * (fp8 ? 1 : 2)};
    const cuuint32_t box[2] = {box_cols, box_rows};
    const cuuint32_t estr[2] = {1, 1};
    const CUtensorMapDataType dt = fp8    ? CU_TENSOR_MAP_DATA_TYPE_UINT8
                                   : bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                          : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
    CUresult r = fn(map, dt, 2, const_cast<void*>(ptr), dims, strides,
                    box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS)
        return fail(GEMM_F16_ERR_CUDA, "cuTensorMapEncodeTiled failed (CUresult %d) for %llux%llu",
                    (int)r, (unsigned long long)rows, (unsigned long long)cols);
    return GEMM_F16_OK;
}

// Block scales in the tiled layout (mx_sf_offset) of a `rows` x K operand, viewed as a 3-D
// tensor of 32-bit words {128 words = one 512-byte chunk, K-block groups, 128-row groups}; a box
// is `chunks` consecutive row groups of one K-block group.  Row groups past the end read as zero.
int make_sf_map(CUtensorMap* map, const void* ptr, uint64_t rows, uint64_t K, uint32_t chunks)
{
    auto fn = encode_fn();
    if (!fn) return fail(GEMM_F16_ERR_CUDA, "cuTensorMapEncodeTiled is not available");
    const uint64_t kgroups = gf16::mx_k_groups(static_cast<uint32_t>(K / 32));
    const cuuint64_t dims[3] = {128, kgroups, (rows + 127) / 128};
    const cuuint64_t strides[2] = {512, kgroups * 512};
    const cuuint32_t box[3] = {128, 1, chunks};
    const cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT32, 3, const_cast<void*>(ptr), dims, strides,
                    box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS)
        return fail(GEMM_F16_ERR_CUDA, "cuTensorMapEncodeTiled failed (CUresult %d) for the "
                    "scales of %llu rows, K=%llu", (int)r, (unsigned long long)rows,
                    (unsigned long long)K);
    return GEMM_F16_OK;
}

// Small per-thread cache of encoded descriptors, keyed by everything they encode.
struct MapKey {
    const void* a;
    const void* b;
    const void* d;
    int64_t M, N, K;
    int variant;
    int device;
    int dtype = 0;           // GEMM_F16_DTYPE_* of the 16-bit operands / output
    const void* sfa = nullptr;  // block-scaled path: scale buffers (else null)
    const void* sfb = nullptr;
    bool operator==(const MapKey& o) const
    {
        return a == o.a && b == o.b && d == o.d && M == o.M && N == o.N && K == o.K &&
               variant == o.variant && device == o.device && dtype == o.dtype && sfa == o.sfa &&
               sfb == o.sfb;
    }
};

struct MapEntry {
    MapKey key;
    CUtensorMap ma, mb, md, msfa, msfb;
    CUtensorMap mbh;   // B in boxes of half the rows (half-width tail items; 16-bit path)
    bool valid;
};

constexpr int kCacheSize = 8;
thread_local MapEntry t_cache[kCacheSize];
thread_local int t_cache_next = 0;

// Descriptors of one launch.  mx: FP8 operands (8-bit codes, 128-element boxes) plus the two
// scale maps, B's boxes holding sfb_chunks row groups.
int get_maps(const MapKey& k, uint32_t a_box_rows, uint32_t b_box_rows, bool need_d,
             const MapEntry** out, bool mx = false, uint32_t sfb_chunks = 0)
{
    for (auto& e : t_cache) {
        if (e.valid && e.key == k) {
            *out = &e;
            return GEMM_F16_OK;
        }
    }
    MapEntry& e = t_cache[t_cache_next];
    t_cache_next = (t_cache_next + 1) % kCacheSize;
    e.valid = false;
    int rc;
    const bool bf = k.dtype == GEMM_F16_DTYPE_BF16;
    const uint32_t box_k = mx ? 128 : 64;
    if ((rc = make_map(&e.ma, k.a, k.M, k.K, a_box_rows, box_k, !mx && bf, mx)) != GEMM_F16_OK)
        return rc;
    if ((rc = make_map(&e.mb, k.b, k.N, k.K, b_box_rows, box_k, !mx && bf, mx)) != GEMM_F16_OK)
        return rc;
    if (!mx && b_box_rows >= 16) {
        if ((rc = make_map(&e.mbh, k.b, k.N, k.K, b_box_rows / 2, box_k, bf)) != GEMM_F16_OK)
            return rc;
    } else {
        std::memset(&e.mbh, 0, sizeof(e.mbh));
    }
    if (need_d) {
        if ((rc = make_map(&e.md, k.d, k.M, k.N, 128, 64, bf)) != GEMM_F16_OK) return rc;
    } else {
        std::memset(&e.md, 0, sizeof(e.md));
    }
    if (mx) {
        if ((rc = make_sf_map(&e.msfa, k.sfa, k.M, k.K, 1)) != GEMM_F16_OK) return rc;
        if ((rc = make_sf_map(&e.msfb, k.sfb, k.N, k.K, sfb_chunks)) != GEMM_F16_OK) return rc;
    } else {
        std::memset(&e.msfa, 0, sizeof(e.msfa));
        std::memset(&e.msfb, 0, sizeof(e.msfb));
    }
    e.key = k;
    e.valid = true;
    *out = &e;
    return GEMM_F16_OK;
}

// ---- launches --------------------------------------------------------------------------------
// The tile variant's N tile: the narrowest of 16, 32, 64 whose grid still fits one wave of
// `sms` CTAs, else 128.  A small D then spreads over more SMs, each loading and storing less.
int tile_bn_for(int64_t M, int64_t N, int sms)
{
    for (int bn = 16; bn < 128; bn *= 2)
        if (cdiv(M, 128) * cdiv(N, bn) <= sms) return bn;
    return 128;
}

template <uint32_t kBN>
int launch_tile(const void* A, const void* B, void* D, int64_t M, int64_t N, int64_t K,
                cudaStream_t stream, DeviceState& d, int dev)
{
    using C = gf16::TileCfg<kBN>;
    // kernel slots 56 .. 59 and descriptor-cache keys 116 .. 228, one per N tile
    constexpr int slot = kBN == 16 ? 56 : kBN == 32 ? 57 : kBN == 64 ? 58 : 59;
    int rc = ensure_smem(d, slot, gf16::gemm_tile_kernel<kBN>, C::SMEM_ALLOC);
    if (rc != GEMM_F16_OK) return rc;
    const MapEntry* maps = nullptr;
    MapKey key{A, B, D, M, N, K, 100 + static_cast<int>(kBN), dev};
    if ((rc = get_maps(key, 128, kBN, false, &maps)) != GEMM_F16_OK) return rc;
    const dim3 grid(static_cast<uint32_t>(cdiv(N, kBN)), static_cast<uint32_t>(cdiv(M, 128)));
    if (grid.y > 65535u) return fail(GEMM_F16_ERR_UNSUPPORTED, "M too large for the tile variant");
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(C::THREADS);
    cfg.dynamicSmemBytes = C::SMEM_ALLOC;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    cfg.attrs = attr;
    cfg.numAttrs = 0;
    if (pdl_setting()) {
        // The kernel waits (griddepcontrol.wait) before its first global-memory access.
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.numAttrs = 1;
    }
    cudaError_t e = cudaLaunchKernelEx(&cfg, gf16::gemm_tile_kernel<kBN>, maps->ma, maps->mb,
                                       static_cast<uint16_t*>(D), (uint32_t)M, (uint32_t)N,
                                       (uint32_t)cdiv(K, 64), wait_timeout_ns(), debug_flags());
    if (e != cudaSuccess) return cuda_fail(e, "cudaLaunchKernelEx(gemm_tile_kernel)");
    return GEMM_F16_OK;
}

// Units that share the stream-K tail of R tiles: at most 3 per tile, so a tile has at most
// 4 contributors (gf16::kMaxContrib: the piece that finishes a tile adds up to 3 others).
int64_t sk_units_for(int64_t R, int64_t U)
{
    return R * 3 < U ? R * 3 : U;
}

// Stream-K tail size for T tiles of KB k-blocks on U units: the tiles of the last, partial
// wave (all tiles when T < U), or 0 when the tail is nearly a full wave or the per-unit pieces
// would be tiny.
int64_t sk_tail_tiles(int64_t T, int64_t U, int64_t KB)
{
    if (T <= 0 || U <= 0) return 0;
    const int64_t R = T < U ? T : T % U;
    if (R == 0) return 0;
    if (R * 10 > U * 9) return 0;   // the last wave is at least 90% full already
    if (R * KB < 4 * sk_units_for(R, U)) return 0;   // under 4 k-blocks per unit
    return R;
}

// Half-width tail: the tiles of the last, partial wave (all of them when there are fewer tiles
// than units) each become two items of half the columns, when those fit in one wave (2 R <= U).
// The last wave then takes about half a tile's time.  0: none.
int64_t half_tail_tiles(int64_t T, int64_t U)
{
    if (T <= 0 || U <= 0) return 0;
    const int64_t R = T < U ? T : T % U;
    return R > 0 && 2 * R <= U ? R : 0;
}

// GEMM_F16_HALF_TAIL=0 (read once per process) turns the half-width tail off, for comparison.
bool half_tail_setting()
{
    static const bool v = [] {
        const char* s = std::getenv("GEMM_F16_HALF_TAIL");
        return !(s && s[0] == '0');
    }();
    return v;
}

// Workspace layout: [header, gf16::kSkHeaderBytes][partial sums: units x cta_group x 128 x BN
// fp32].  The header must be zero when a workspace is first used and the kernel keeps it so
// (see gf16::kSkHeaderBytes).  A caller's workspace has its header cleared with
// cudaMemsetAsync on the launch's stream before each launch, so it needs no initialising; the
// library's own fixed array (gemm_f16_nt_noalloc) starts at zero and skips that clear.
size_t ws_bytes_for(int64_t units, int cta_group, int block_n)
{
    return gf16::kSkHeaderBytes + static_cast<size_t>(units) * cta_group * 128u * block_n * 4u;
}

// Set while gemm_f16_nt_noalloc runs a launch on its fixed array (see ws_bytes_for).
thread_local bool t_ws_kept_clean = false;

// Whether launches given a workspace run the stream-K tail (gemm_f16_set_stream_k).  Off by
// default: measured on GB300, it was slower than the data-parallel schedule on every workload
// (a CTA parks 128 KB of fp32 partial sums at about 25 bytes per cycle, and the finishing CTA
// reads them back, which costs more than the idle part of the last wave).
std::atomic<int> g_stream_k{0};

// Epilogue options of a launch: element type, bias (N elements of that type, or null) and
// activation.
struct EpiOpts {
    int dtype = GEMM_F16_DTYPE_F16;
    const void* bias = nullptr;
    int act = GEMM_F16_ACT_NONE;
};

// Block-scaled operands of a launch: the two tiled scale buffers and the element formats.
struct MxOpts {
    const void* sfa = nullptr;
    const void* sfb = nullptr;
    int fmt_a = GEMM_MXF8_E4M3;
    int fmt_b = GEMM_MXF8_E4M3;
};

template <int kCtaGroup, int kBlockN, int kStages, bool kTmaStore, bool kBf16 = false,
          bool kMx = false, int kAccBufs = 2, int kDBufs = 2>
int launch_ws(int variant, const void* A, const void* B, void* D, int64_t M, int64_t N, int64_t K,
              cudaStream_t stream, DeviceState& d, int dev, void* workspace = nullptr,
              size_t workspace_bytes = 0, size_t* bytes_needed = nullptr,
              const EpiOpts& epi = EpiOpts{}, const MxOpts& mx = MxOpts{})
{
    using C = gf16::WsCfg<kCtaGroup, kBlockN, kStages, kTmaStore, kMx, kAccBufs, kDBufs>;
    auto kernel = gf16::gemm_ws_kernel<kCtaGroup, kBlockN, kStages, kTmaStore, kBf16, kMx,
                                       kAccBufs, kDBufs>;
    const int slot = kMx ? kMxSlot0 + 2 * variant + (kBf16 ? 1 : 0)
                         : variant + (kBf16 ? GEMM_F16_NUM_VARIANTS : 0);
    int rc = ensure_smem(d, slot, kernel, C::SMEM_ALLOC);
    if (rc != GEMM_F16_OK) return rc;

    const int64_t num_m = cdiv(M, C::MMA_M);
    const int64_t num_n = cdiv(N, C::BN);
    const int64_t tiles = num_m * num_n;
    if (tiles > 0x7FFFFFFFll) return fail(GEMM_F16_ERR_UNSUPPORTED, "too many tiles");

    cudaLaunchConfig_t cfg{};
    cudaLaunchAttribute attr[2];
    cfg.blockDim = dim3(C::THREADS);
    cfg.dynamicSmemBytes = C::SMEM_ALLOC;
    cfg.stream = stream;
    int64_t units = d.sms;
    if constexpr (kCtaGroup == 2) {
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = 2;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        {
            std::lock_guard<std::mutex> lk(g_mu);
            if (d.pair_clusters[slot] == 0) {
                cfg.gridDim = dim3(2 * (d.sms / 2));
                int n = 0;
                cudaError_t e = cudaOccupancyMaxActiveClusters(&n, kernel, &cfg);
                if (e != cudaSuccess) return cuda_fail(e, "cudaOccupancyMaxActiveClusters");
                if (n < 1) return fail(GEMM_F16_ERR_CUDA, "no CTA pair fits on this device");
                d.pair_clusters[slot] = n;
            }
            units = d.pair_clusters[slot];
        }
    } else {
        cfg.attrs = attr;
        cfg.numAttrs = 0;
    }
    if (pdl_setting()) {
        // The kernel waits (griddepcontrol.wait) before its first global-memory access, so the
        // launch may overlap the end of the kernel before it on the stream.
        attr[cfg.numAttrs].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[cfg.numAttrs].val.programmaticStreamSerializationAllowed = 1;
        ++cfg.numAttrs;
    }
    const int64_t KB = cdiv(K, C::BLOCK_K);
    // Stream-K tail: all units take part; otherwise no more units than tiles.
    int64_t R = g_stream_k.load(std::memory_order_relaxed) ? sk_tail_tiles(tiles, units, KB) : 0;
    // one flag per (tail tile, contributor, CTA) in each of the header's two flag regions
    if (R * gf16::kMaxContrib * kCtaGroup > gf16::kSkFlagWords) R = 0;
    const size_t need = R ? ws_bytes_for(units, kCtaGroup, kBlockN) : 0;
    if (bytes_needed) {
        *bytes_needed = need;
        return GEMM_F16_OK;
    }
    const MapEntry* maps = nullptr;
    MapKey key{A, B, D, M, N, K, kMx ? -1 - variant : variant, dev,
               kBf16 ? GEMM_F16_DTYPE_BF16 : GEMM_F16_DTYPE_F16, mx.sfa, mx.sfb};
    if ((rc = get_maps(key, 128, C::B_ROWS, kTmaStore, &maps, kMx, C::SFB_CHUNKS)) != GEMM_F16_OK)
        return rc;
    const uint32_t mx_idesc =
        kMx ? gf16::make_idesc_mx(C::MMA_M, C::BN, static_cast<uint32_t>(mx.fmt_a),
                                  static_cast<uint32_t>(mx.fmt_b))
            : 0u;
    if (R && (workspace == nullptr || workspace_bytes < need ||
              (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0))
        R = 0;  // no usable workspace: plain data-parallel schedule
    // Without a stream-K tail, the last partial wave may run as half-width items (16-bit path;
    // the epilogue stores 64-column chunks, so half a tile must be a whole number of them).
    const int64_t H = (!kMx && R == 0 && (C::BN / 2) % 64 == 0 && half_tail_setting())
                          ? half_tail_tiles(tiles, units)
                          : 0;
    const int64_t units_used = R ? units
                               : H ? (tiles == H ? 2 * H : units)
                                   : (tiles < units ? tiles : units);
    cfg.gridDim = dim3(static_cast<uint32_t>(kCtaGroup * units_used));
    // Pipeline positions are 32-bit counters over a unit's k-block iterations.
    if ((cdiv(tiles - R, units_used) + 1) * KB >= (int64_t(1) << 31))
        return fail(GEMM_F16_ERR_UNSUPPORTED, "problem too large for one launch (M=%lld N=%lld "
                    "K=%lld)", (long long)M, (long long)N, (long long)K);
    uint32_t* ws_hdr = nullptr;
    float* ws_part = nullptr;
    if (R) {
        ws_hdr = static_cast<uint32_t*>(workspace);
        ws_part = reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) + gf16::kSkHeaderBytes);
        if (!t_ws_kept_clean) {
            cudaError_t e = cudaMemsetAsync(ws_hdr, 0, gf16::kSkHeaderBytes, stream);
            if (e != cudaSuccess) return cuda_fail(e, "cudaMemsetAsync(stream-K header)");
        }
    }
    cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, maps->ma, maps->mb, maps->md,
                                       static_cast<uint16_t*>(D),
                                       (uint32_t)M, (uint32_t)N,
                                       (uint32_t)num_m, (uint32_t)num_n, (uint32_t)KB,
                                       group_m_for(C::MMA_M, K, C::ELEM_BYTES, d.l2_bytes),
                                       wait_timeout_ns(), l2_hint_setting(),
                                       ws_part, ws_hdr, (uint32_t)R,
                                       (uint32_t)(R ? sk_units_for(R, units_used) : units_used),
                                       static_cast<const uint16_t*>(epi.bias),
                                       static_cast<uint32_t>(epi.act), debug_flags(),
                                       maps->msfa, maps->msfb, mx_idesc, maps->mbh,
                                       static_cast<uint32_t>(H));
    if (e != cudaSuccess) return cuda_fail(e, "cudaLaunchKernelEx(gemm_ws_kernel)");
    return GEMM_F16_OK;
}

int check_args(const void* A, const void* B, void* D, int64_t M, int64_t N, int64_t K)
{
    const int64_t lim = 0x7FFFFFFFll;
    if (M < 0 || N < 0 || K < 0)
        return fail(GEMM_F16_ERR_INVALID_ARG, "negative size (M=%lld N=%lld K=%lld)", (long long)M,
                    (long long)N, (long long)K);
    if (M > lim || N > lim || K > lim)
        return fail(GEMM_F16_ERR_INVALID_ARG, "size above 2^31-1 (M=%lld N=%lld K=%lld)",
                    (long long)M, (long long)N, (long long)K);
    if (M == 0 || N == 0) return GEMM_F16_OK;
    if (D == nullptr) return fail(GEMM_F16_ERR_INVALID_ARG, "D is null");
    if (K > 0 && (A == nullptr || B == nullptr))
        return fail(GEMM_F16_ERR_INVALID_ARG, "A or B is null");
    if (K % 8 != 0)
        return fail(GEMM_F16_ERR_UNSUPPORTED, "K=%lld is not a multiple of 8", (long long)K);
    if (N % 8 != 0)
        return fail(GEMM_F16_ERR_UNSUPPORTED, "N=%lld is not a multiple of 8", (long long)N);
    auto misaligned = [](const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) != 0; };
    if (misaligned(D) || (K > 0 && (misaligned(A) || misaligned(B))))
        return fail(GEMM_F16_ERR_UNSUPPORTED, "A, B and D must be 16-byte aligned");
    return GEMM_F16_OK;
}

int run(const void* A, const void* B, void* D, int64_t M, int64_t N, int64_t K,
        cudaStream_t stream, int variant, void* ws = nullptr, size_t ws_bytes = 0,
        size_t* bytes_needed = nullptr, const EpiOpts& epi = EpiOpts{})
{
    t_last_error.clear();
    if (bytes_needed) *bytes_needed = 0;
    if (variant < 0 || variant >= GEMM_F16_NUM_VARIANTS)
        return fail(GEMM_F16_ERR_INVALID_ARG, "unknown variant %d", variant);
    int rc = bytes_needed ? GEMM_F16_OK : check_args(A, B, D, M, N, K);
    if (rc != GEMM_F16_OK) return rc;
    if (M < 0 || N < 0 || K < 0) return fail(GEMM_F16_ERR_INVALID_ARG, "negative size");
    if (M == 0 || N == 0) return GEMM_F16_OK;
    if (bytes_needed && K == 0) return GEMM_F16_OK;
    if (K == 0) {
        cudaError_t e = cudaMemsetAsync(D, 0, static_cast<size_t>(M) * N * 2, stream);
        return e == cudaSuccess ? GEMM_F16_OK : cuda_fail(e, "cudaMemsetAsync");
    }
    DeviceState* d = nullptr;
    if ((rc = device_state(&d)) != GEMM_F16_OK) return rc;
    int dev = 0;
    cudaGetDevice(&dev);
    const bool plain = epi.dtype == GEMM_F16_DTYPE_F16 && epi.bias == nullptr &&
                       epi.act == GEMM_F16_ACT_NONE;
    if (variant == GEMM_F16_VARIANT_AUTO) {
        variant = choose_variant(M, N, K, d->sms);
        // the one-tile kernel has no bf16 / fused-epilogue form
        if (!plain && variant == GEMM_F16_VARIANT_TILE) variant = GEMM_F16_VARIANT_WS_128x128;
    }
    if (!plain) {
        if (epi.dtype != GEMM_F16_DTYPE_F16 && epi.dtype != GEMM_F16_DTYPE_BF16)
            return fail(GEMM_F16_ERR_INVALID_ARG, "unknown dtype %d", epi.dtype);
        if (epi.act < GEMM_F16_ACT_NONE || epi.act > GEMM_F16_ACT_GELU)
            return fail(GEMM_F16_ERR_INVALID_ARG, "unknown activation %d", epi.act);
        if (epi.bias != nullptr && (reinterpret_cast<uintptr_t>(epi.bias) & 15u) != 0)
            return fail(GEMM_F16_ERR_UNSUPPORTED, "bias must be 16-byte aligned");
        if (K == 0)
            return fail(GEMM_F16_ERR_UNSUPPORTED, "K == 0 with a fused epilogue is not supported");
        const bool bf = epi.dtype == GEMM_F16_DTYPE_BF16;
        switch (variant) {
        case GEMM_F16_VARIANT_WS_128x256:
            return bf ? launch_ws<1, 256, 4, true, true>(variant, A, B, D, M, N, K, stream, *d, dev,
                                                         ws, ws_bytes, bytes_needed, epi)
                      : launch_ws<1, 256, 4, true>(variant, A, B, D, M, N, K, stream, *d, dev, ws,
                                                   ws_bytes, bytes_needed, epi);
        case GEMM_F16_VARIANT_WS_PAIR:
            return bf ? launch_ws<2, 256, 6, true, true>(variant, A, B, D, M, N, K, stream, *d, dev,
                                                         ws, ws_bytes, bytes_needed, epi)
                      : launch_ws<2, 256, 6, true>(variant, A, B, D, M, N, K, stream, *d, dev, ws,
                                                   ws_bytes, bytes_needed, epi);
        case GEMM_F16_VARIANT_WS_128x128:
            return bf ? launch_ws<1, 128, 6, true, true>(variant, A, B, D, M, N, K, stream, *d, dev,
                                                         ws, ws_bytes, bytes_needed, epi)
                      : launch_ws<1, 128, 6, true>(variant, A, B, D, M, N, K, stream, *d, dev, ws,
                                                   ws_bytes, bytes_needed, epi);
        case GEMM_F16_VARIANT_WS_PAIR_256x192:
            return bf ? launch_ws<2, 192, 6, true, true>(variant, A, B, D, M, N, K, stream, *d, dev,
                                                         ws, ws_bytes, bytes_needed, epi)
                      : launch_ws<2, 192, 6, true>(variant, A, B, D, M, N, K, stream, *d, dev, ws,
                                                   ws_bytes, bytes_needed, epi);
        default:
            return fail(GEMM_F16_ERR_UNSUPPORTED,
                        "variant %d has no bf16 / fused-epilogue form (use 0, 2, 3, 4 or 6)",
                        variant);
        }
    }
    switch (variant) {
    case GEMM_F16_VARIANT_TILE:
        if (bytes_needed) return GEMM_F16_OK;
        switch (tile_bn_for(M, N, d->sms)) {
        case 16: return launch_tile<16>(A, B, D, M, N, K, stream, *d, dev);
        case 32: return launch_tile<32>(A, B, D, M, N, K, stream, *d, dev);
        case 64: return launch_tile<64>(A, B, D, M, N, K, stream, *d, dev);
        default: return launch_tile<128>(A, B, D, M, N, K, stream, *d, dev);
        }
    case GEMM_F16_VARIANT_WS_128x256:
        return launch_ws<1, 256, 4, true>(variant, A, B, D, M, N, K, stream, *d, dev, ws,
                                          ws_bytes, bytes_needed);
    case GEMM_F16_VARIANT_WS_PAIR:
        return launch_ws<2, 256, 6, true>(variant, A, B, D, M, N, K, stream, *d, dev, ws,
                                          ws_bytes, bytes_needed);
    case GEMM_F16_VARIANT_WS_128x128:
        return launch_ws<1, 128, 6, true>(variant, A, B, D, M, N, K, stream, *d, dev, ws,
                                          ws_bytes, bytes_needed);
    case GEMM_F16_VARIANT_WS_PAIR_DIRECT:
        return launch_ws<2, 256, 7, false>(variant, A, B, D, M, N, K, stream, *d, dev, ws,
                                           ws_bytes, bytes_needed);
    case GEMM_F16_VARIANT_WS_PAIR_256x192:
        return launch_ws<2, 192, 6, true>(variant, A, B, D, M, N, K, stream, *d, dev, ws,
                                          ws_bytes, bytes_needed);
    default:
        return fail(GEMM_F16_ERR_INVALID_ARG, "unknown variant %d", variant);
    }
}

// ---- scratch for callers that cannot allocate -------------------------------------------------
// gemm_f16_nt_noalloc runs the stream-K schedule with its workspace in this fixed array instead
// of caller memory.  The array exists on every device that loads the library, for the life of
// the process.  Host code must not use its name as a device address (on the host it is only a
// stand-in); the device address is looked up once per device with cudaGetSymbolAddress.
constexpr size_t kNoAllocScratchBytes = size_t(40) << 20;   // 40 MiB
static __device__ __align__(256) uint8_t g_noalloc_scratch[kNoAllocScratchBytes];

std::mutex g_noalloc_mu;
void* g_noalloc_ptr[kMaxDevices] = {};

// Device address of g_noalloc_scratch on the current device (looked up on first use).
int noalloc_scratch(void** out)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    if (dev < 0 || dev >= kMaxDevices) return fail(GEMM_F16_ERR_CUDA, "device %d out of range", dev);
    std::lock_guard<std::mutex> lk(g_noalloc_mu);
    if (g_noalloc_ptr[dev] == nullptr) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(no-alloc scratch)");
        if (p == nullptr) return fail(GEMM_F16_ERR_CUDA, "no device address for the scratch array");
        g_noalloc_ptr[dev] = p;
    }
    *out = g_noalloc_ptr[dev];
    return GEMM_F16_OK;
}

// ---- block-scaled FP8 (MX) ---------------------------------------------------------------------
// 128x128 tiles on one CTA (5-stage ring) and 256x128 tiles on a CTA pair (7 stages).  Both keep
// two 128-column accumulators, so the scale-factor ring fits beside them in tensor memory.
using MxCta = gf16::WsCfg<1, 128, 5, true, true>;
using MxPair = gf16::WsCfg<2, 128, 7, true, true>;
// 256x192 on a CTA pair: two 192-column accumulators and a 6-slot scale ring (456 columns).  An
// N tile that starts 64 rows into a 128-row scale group reads B's scales 2 columns further on.
// (A 7th stage in exchange for a single staging buffer measured 4.7% more cycles on 8192^3.)
using MxPair192 = gf16::WsCfg<2, 192, 6, true, true>;
// 256x256 on a CTA pair with one 256-column accumulator (so the scales fit beside it) and a
// 6-slot scale ring: the epilogue frees the accumulator before it stores, so one staging buffer
// is enough and its 16 KB go to a sixth pipeline stage.
using MxPair256 = gf16::WsCfg<2, 256, 6, true, true, 1, 1>;

// Measured on GB300 (bench.py --sweep --sweep-mx): the single-accumulator 256x256 pair is the
// fastest at 2048^3 (13.2 us against 15.2 us for 128x128), 8192^3 and the MLP shape, and within
// 1% of 256x192 on 3000x5000x1056; one 128x128 tile is faster on a single CTA.
int choose_mx_variant(int64_t M, int64_t N, int64_t /*K*/, int /*num_sms*/)
{
    if (M <= 128 || N <= 128) return GEMM_MXF8_VARIANT_128x128;
    return GEMM_MXF8_VARIANT_PAIR_256x256;
}

int64_t mx_scale_bytes(int64_t rows, int64_t K)
{
    if (rows < 0 || K < 0 || K % 32 != 0) return -1;
    return cdiv(rows, 128) * static_cast<int64_t>(gf16::mx_k_groups(static_cast<uint32_t>(K / 32))) *
           512;
}

int check_mx_args(const void* A, const void* B, const void* SFA, const void* SFB, void* D,
                  int64_t M, int64_t N, int64_t K, int fmt_a, int fmt_b, const EpiOpts& epi)
{
    int rc = check_args(A, B, D, M, N, K);
    if (rc != GEMM_F16_OK) return rc;
    if (fmt_a < GEMM_MXF8_E4M3 || fmt_a > GEMM_MXF8_E5M2 || fmt_b < GEMM_MXF8_E4M3 ||
        fmt_b > GEMM_MXF8_E5M2)
        return fail(GEMM_F16_ERR_INVALID_ARG, "unknown FP8 format (A %d, B %d)", fmt_a, fmt_b);
    if (epi.dtype != GEMM_F16_DTYPE_F16 && epi.dtype != GEMM_F16_DTYPE_BF16)
        return fail(GEMM_F16_ERR_INVALID_ARG, "unknown output dtype %d", epi.dtype);
    if (epi.act < GEMM_F16_ACT_NONE || epi.act > GEMM_F16_ACT_GELU)
        return fail(GEMM_F16_ERR_INVALID_ARG, "unknown activation %d", epi.act);
    if (M == 0 || N == 0) return GEMM_F16_OK;
    if (K % 32 != 0)
        return fail(GEMM_F16_ERR_UNSUPPORTED, "K=%lld is not a multiple of the 32-element scale "
                    "block", (long long)K);
    auto misaligned = [](const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) != 0; };
    if (K > 0 && (SFA == nullptr || SFB == nullptr))
        return fail(GEMM_F16_ERR_INVALID_ARG, "SFA or SFB is null");
    if (K > 0 && (misaligned(SFA) || misaligned(SFB)))
        return fail(GEMM_F16_ERR_UNSUPPORTED, "SFA and SFB must be 16-byte aligned");
    if (epi.bias != nullptr && misaligned(epi.bias))
        return fail(GEMM_F16_ERR_UNSUPPORTED, "bias must be 16-byte aligned");
    return GEMM_F16_OK;
}

int run_mx(const void* A, const void* B, const void* SFA, const void* SFB, void* D, int64_t M,
           int64_t N, int64_t K, int fmt_a, int fmt_b, const EpiOpts& epi, int variant, void* ws,
           size_t ws_bytes, size_t* bytes_needed, cudaStream_t stream)
{
    t_last_error.clear();
    if (bytes_needed) *bytes_needed = 0;
    if (variant < 0 || variant >= GEMM_MXF8_NUM_VARIANTS)
        return fail(GEMM_F16_ERR_INVALID_ARG, "unknown block-scaled variant %d", variant);
    if (M < 0 || N < 0 || K < 0) return fail(GEMM_F16_ERR_INVALID_ARG, "negative size");
    int rc = bytes_needed ? GEMM_F16_OK
                          : check_mx_args(A, B, SFA, SFB, D, M, N, K, fmt_a, fmt_b, epi);
    if (rc != GEMM_F16_OK) return rc;
    if (M == 0 || N == 0) return GEMM_F16_OK;
    if (K == 0) {
        if (bytes_needed) return GEMM_F16_OK;
        if (epi.bias != nullptr || epi.act != GEMM_F16_ACT_NONE)
            return fail(GEMM_F16_ERR_UNSUPPORTED, "K == 0 with a fused epilogue is not supported");
        cudaError_t e = cudaMemsetAsync(D, 0, static_cast<size_t>(M) * N * 2, stream);
        return e == cudaSuccess ? GEMM_F16_OK : cuda_fail(e, "cudaMemsetAsync");
    }
    DeviceState* d = nullptr;
    if ((rc = device_state(&d)) != GEMM_F16_OK) return rc;
    int dev = 0;
    cudaGetDevice(&dev);
    if (variant == GEMM_MXF8_VARIANT_AUTO) variant = choose_mx_variant(M, N, K, d->sms);
    const MxOpts mx{SFA, SFB, fmt_a, fmt_b};
    const bool bf = epi.dtype == GEMM_F16_DTYPE_BF16;
    switch (variant) {
    case GEMM_MXF8_VARIANT_128x128:
        return bf ? launch_ws<1, 128, 5, true, true, true>(variant, A, B, D, M, N, K, stream, *d,
                                                           dev, ws, ws_bytes, bytes_needed, epi, mx)
                  : launch_ws<1, 128, 5, true, false, true>(variant, A, B, D, M, N, K, stream, *d,
                                                            dev, ws, ws_bytes, bytes_needed, epi,
                                                            mx);
    case GEMM_MXF8_VARIANT_PAIR_256x128:
        return bf ? launch_ws<2, 128, 7, true, true, true>(variant, A, B, D, M, N, K, stream, *d,
                                                           dev, ws, ws_bytes, bytes_needed, epi, mx)
                  : launch_ws<2, 128, 7, true, false, true>(variant, A, B, D, M, N, K, stream, *d,
                                                            dev, ws, ws_bytes, bytes_needed, epi,
                                                            mx);
    case GEMM_MXF8_VARIANT_PAIR_256x192:
        return bf ? launch_ws<2, 192, 6, true, true, true>(variant, A, B, D, M, N, K, stream, *d,
                                                           dev, ws, ws_bytes, bytes_needed, epi, mx)
                  : launch_ws<2, 192, 6, true, false, true>(variant, A, B, D, M, N, K, stream, *d,
                                                            dev, ws, ws_bytes, bytes_needed, epi,
                                                            mx);
    case GEMM_MXF8_VARIANT_PAIR_256x256:
        return bf ? launch_ws<2, 256, 6, true, true, true, 1, 1>(variant, A, B, D, M, N, K,
                                                                 stream, *d, dev, ws, ws_bytes,
                                                                 bytes_needed, epi, mx)
                  : launch_ws<2, 256, 6, true, false, true, 1, 1>(variant, A, B, D, M, N, K,
                                                                  stream, *d, dev, ws, ws_bytes,
                                                                  bytes_needed, epi, mx);
    default:
        return fail(GEMM_F16_ERR_INVALID_ARG, "unknown block-scaled variant %d", variant);
    }
}

}  // namespace

// ================================ C ABI ======================================================
extern "C" {

int gemm_f16_nt(const void* A, const void* B, void* D, int64_t M, int64_t N, int64_t K,
                cudaStream_t stream)
{
    return run(A, B, D, M, N, K, stream, GEMM_F16_VARIANT_AUTO);
}

int gemm_f16_nt_variant(const void* A, const void* B, void* D, int64_t M, int64_t N, int64_t K,
                        cudaStream_t stream, int variant)
{
    return run(A, B, D, M, N, K, stream, variant);
}

int gemm_f16_nt_ws(const void* A, const void* B, void* D, int64_t M, int64_t N, int64_t K,
                   void* workspace, size_t workspace_bytes, cudaStream_t stream)
{
    return run(A, B, D, M, N, K, stream, GEMM_F16_VARIANT_AUTO, workspace, workspace_bytes);
}

int gemm_f16_nt_ex(const void* A, const void* B, void* D, int64_t M, int64_t N, int64_t K,
                   int variant, void* workspace, size_t workspace_bytes, cudaStream_t stream)
{
    return run(A, B, D, M, N, K, stream, variant, workspace, workspace_bytes);
}

int gemm_f16_nt_fused(const void* A, const void* B, void* D, int64_t M, int64_t N, int64_t K,
                      int dtype, const void* bias, int activation, int variant, void* workspace,
                      size_t workspace_bytes, cudaStream_t stream)
{
    EpiOpts epi;
    epi.dtype = dtype;
    epi.bias = bias;
    epi.act = activation;
    return run(A, B, D, M, N, K, stream, variant, workspace, workspace_bytes, nullptr, epi);
}

int gemm_f16_nt_noalloc(const void* A, const void* B, void* D, int64_t M, int64_t N, int64_t K,
                        cudaStream_t stream)
{
    t_last_error.clear();
    int rc = check_args(A, B, D, M, N, K);
    if (rc != GEMM_F16_OK) return rc;
    if (M == 0 || N == 0) return GEMM_F16_OK;
    size_t need = 0;
    if (K > 0) {
        rc = run(nullptr, nullptr, nullptr, M, N, K, nullptr, GEMM_F16_VARIANT_AUTO, nullptr, 0,
                 &need);
        if (rc != GEMM_F16_OK) return rc;
    }
    // A stream-K workspace larger than the fixed array (a GPU with many more SMs than a GB300)
    // is not offered: the launch then takes the plain data-parallel schedule, which needs none.
    if (need > kNoAllocScratchBytes) need = 0;
    void* scratch = nullptr;
    if (need > 0 && (rc = noalloc_scratch(&scratch)) != GEMM_F16_OK) return rc;
    // The array's stream-K header starts at zero and every launch leaves it consistent, so
    // the launch needs no clearing copy before it (which would also break the overlap of
    // consecutive launches).
    t_ws_kept_clean = true;
    rc = run(A, B, D, M, N, K, stream, GEMM_F16_VARIANT_AUTO, scratch,
             need > 0 ? kNoAllocScratchBytes : 0);
    t_ws_kept_clean = false;
    return rc;
}

size_t gemm_f16_noalloc_scratch_bytes(void) { return kNoAllocScratchBytes; }

int gemm_f16_workspace_bytes(int64_t M, int64_t N, int64_t K, int variant, size_t* bytes)
{
    if (!bytes) return fail(GEMM_F16_ERR_INVALID_ARG, "bytes is null");
    return run(nullptr, nullptr, nullptr, M, N, K, nullptr, variant, nullptr, 0, bytes);
}

int gemm_f16_choose_variant(int64_t M, int64_t N, int64_t K, int num_sms)
{
    return choose_variant(M, N, K, num_sms);
}

int gemm_f16_check_status(cudaStream_t stream, uint32_t* bits)
{
    t_last_error.clear();
    cudaError_t e = cudaStreamSynchronize(stream);
    if (e != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
    uint32_t v = 0;
    e = cudaMemcpyFromSymbol(&v, gf16::gemm_f16_status_word, sizeof(v));
    if (e != cudaSuccess) return cuda_fail(e, "cudaMemcpyFromSymbol(status)");
    if (bits) *bits = v;
    if (v != 0) {
        const uint32_t zero = 0;
        e = cudaMemcpyToSymbol(gf16::gemm_f16_status_word, &zero, sizeof(zero));
        if (e != cudaSuccess) return cuda_fail(e, "cudaMemcpyToSymbol(status)");
        return fail(GEMM_F16_ERR_TIMEOUT, "a kernel gave up a bounded wait (status bits 0x%x)", v);
    }
    return GEMM_F16_OK;
}

const char* gemm_f16_last_error(void) { return t_last_error.c_str(); }

int gemm_f16_set_wait_timeout_ms(uint32_t ms)
{
    if (ms == 0) return fail(GEMM_F16_ERR_INVALID_ARG, "timeout must be at least 1 ms");
    g_timeout_ns.store(static_cast<uint64_t>(ms) * 1000000ull);
    return GEMM_F16_OK;
}

int gemm_f16_set_fault_injection(int mode)
{
    if (mode < 0 || mode > 1) return fail(GEMM_F16_ERR_INVALID_ARG, "unknown injection %d", mode);
    g_debug_flags.store(mode == 1 ? gf16::kDebugNoLoads : 0u);
    return GEMM_F16_OK;
}

int gemm_f16_version(void) { return kVersion; }

int gemm_f16_get_variant_info(int variant, gemm_f16_variant_info* out)
{
    if (!out) return GEMM_F16_ERR_INVALID_ARG;
    return variant_info(variant, out) ? GEMM_F16_OK : GEMM_F16_ERR_INVALID_ARG;
}

uint32_t gemm_f16_idesc(uint32_t M, uint32_t N, uint32_t ab_bf16)
{
    return gf16::make_idesc_f16(M, N, ab_bf16);
}

uint64_t gemm_f16_smem_desc_sw128(uint32_t smem_addr, uint32_t sbo_bytes)
{
    return gf16::make_smem_desc_sw128(smem_addr, sbo_bytes);
}

uint32_t gemm_f16_sw128(uint32_t off) { return gf16::sw128(off); }

void gemm_f16_tile_coord(uint32_t t, uint32_t num_m, uint32_t num_n, uint32_t group,
                         uint32_t* m_blk, uint32_t* n_blk)
{
    const gf16::TileCoord c = gf16::tile_coord(t, num_m, num_n, group);
    if (m_blk) *m_blk = c.m_blk;
    if (n_blk) *n_blk = c.n_blk;
}

uint32_t gemm_f16_raster_group(int64_t mma_m, int64_t K, int64_t elem_bytes, int64_t l2_bytes)
{
    return group_m_for(mma_m, K, elem_bytes, l2_bytes);
}

int64_t gemm_f16_sk_tail_tiles(int64_t tiles, int64_t units, int64_t k_blocks)
{
    return sk_tail_tiles(tiles, units, k_blocks);
}

int gemm_f16_set_stream_k(int enable)
{
    if (enable != 0 && enable != 1)
        return fail(GEMM_F16_ERR_INVALID_ARG, "stream-K switch %d is not 0 or 1", enable);
    g_stream_k.store(enable, std::memory_order_relaxed);
    return GEMM_F16_OK;
}

static gf16::WorkSplit host_split(uint32_t tiles, uint32_t units, uint32_t k_blocks,
                                  uint32_t tail)
{
    const uint32_t S = tail ? static_cast<uint32_t>(sk_units_for(tail, units)) : units;
    return gf16::WorkSplit{tiles, units, k_blocks, tail, S};
}

uint32_t gemm_f16_sk_items(uint32_t tiles, uint32_t units, uint32_t k_blocks, uint32_t tail,
                           uint32_t unit)
{
    return gf16::items_of(host_split(tiles, units, k_blocks, tail), unit);
}

void gemm_f16_sk_item(uint32_t tiles, uint32_t units, uint32_t k_blocks, uint32_t tail,
                      uint32_t unit, uint32_t idx, uint32_t out[5])
{
    const gf16::WorkItem w = gf16::work_item(host_split(tiles, units, k_blocks, tail), unit, idx);
    out[0] = w.tile;
    out[1] = w.kb0;
    out[2] = w.kb1;
    out[3] = w.piece;
    out[4] = w.partial;
}

uint32_t gemm_f16_sk_unit_of(uint32_t tiles, uint32_t units, uint32_t k_blocks, uint32_t tail,
                             uint32_t x)
{
    return gf16::sk_unit_of(host_split(tiles, units, k_blocks, tail), x);
}

int64_t gemm_f16_half_tail_tiles(int64_t tiles, int64_t units)
{
    return half_tail_tiles(tiles, units);
}

static gf16::WorkSplit host_half_split(uint32_t tiles, uint32_t units, uint32_t k_blocks,
                                       uint32_t half)
{
    gf16::WorkSplit w{tiles, units, k_blocks, 0u, units};
    w.H = half;
    return w;
}

uint32_t gemm_f16_half_items(uint32_t tiles, uint32_t units, uint32_t k_blocks, uint32_t half,
                             uint32_t unit)
{
    return gf16::items_of(host_half_split(tiles, units, k_blocks, half), unit);
}

void gemm_f16_half_item(uint32_t tiles, uint32_t units, uint32_t k_blocks, uint32_t half,
                        uint32_t unit, uint32_t idx, uint32_t out[4])
{
    const gf16::WorkItem w =
        gf16::work_item(host_half_split(tiles, units, k_blocks, half), unit, idx);
    out[0] = w.tile;
    out[1] = w.kb0;
    out[2] = w.kb1;
    out[3] = w.half;
}

int gemm_mxf8_nt(const void* A, const void* B, const void* SFA, const void* SFB, void* D,
                 int64_t M, int64_t N, int64_t K, int fmt_a, int fmt_b, int out_dtype,
                 const void* bias, int activation, int variant, void* workspace,
                 size_t workspace_bytes, cudaStream_t stream)
{
    EpiOpts epi;
    epi.dtype = out_dtype;
    epi.bias = bias;
    epi.act = activation;
    return run_mx(A, B, SFA, SFB, D, M, N, K, fmt_a, fmt_b, epi, variant, workspace,
                  workspace_bytes, nullptr, stream);
}

int gemm_mxf8_workspace_bytes(int64_t M, int64_t N, int64_t K, int variant, size_t* bytes)
{
    if (!bytes) return fail(GEMM_F16_ERR_INVALID_ARG, "bytes is null");
    if (K % 32 != 0) return fail(GEMM_F16_ERR_UNSUPPORTED, "K is not a multiple of 32");
    return run_mx(nullptr, nullptr, nullptr, nullptr, nullptr, M, N, K, GEMM_MXF8_E4M3,
                  GEMM_MXF8_E4M3, EpiOpts{}, variant, nullptr, 0, bytes, nullptr);
}

int gemm_mxf8_choose_variant(int64_t M, int64_t N, int64_t K, int num_sms)
{
    return choose_mx_variant(M, N, K, num_sms);
}

int64_t gemm_mxf8_scale_bytes(int64_t rows, int64_t K) { return mx_scale_bytes(rows, K); }

int gemm_mxf8_pack_scales(const void* src, void* dst, int64_t rows, int64_t K,
                          cudaStream_t stream)
{
    t_last_error.clear();
    const int64_t total = mx_scale_bytes(rows, K);
    if (total < 0)
        return fail(GEMM_F16_ERR_INVALID_ARG, "rows=%lld, K=%lld: need rows >= 0 and K a "
                    "non-negative multiple of 32", (long long)rows, (long long)K);
    if (rows > 0x7FFFFFFFll || K > 0x7FFFFFFFll)
        return fail(GEMM_F16_ERR_INVALID_ARG, "size above 2^31-1");
    if (total == 0) return GEMM_F16_OK;
    if (src == nullptr || dst == nullptr) return fail(GEMM_F16_ERR_INVALID_ARG, "null pointer");
    DeviceState* d = nullptr;
    int rc = device_state(&d);
    if (rc != GEMM_F16_OK) return rc;
    const int64_t blocks_needed = cdiv(total, 256);
    const int64_t cap = static_cast<int64_t>(d->sms) * 8;
    const uint32_t grid = static_cast<uint32_t>(blocks_needed < cap ? blocks_needed : cap);
    const uint32_t kb = static_cast<uint32_t>(K / 32);
    gf16::mx_pack_scales_kernel<<<grid, 256, 0, stream>>>(
        static_cast<const uint8_t*>(src), static_cast<uint8_t*>(dst), static_cast<uint64_t>(rows),
        kb, gf16::mx_k_groups(kb), static_cast<uint64_t>(total));
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(e, "launch of mx_pack_scales_kernel");
    return GEMM_F16_OK;
}

uint32_t gemm_mxf8_idesc(uint32_t M, uint32_t N, uint32_t fmt_a, uint32_t fmt_b)
{
    return gf16::make_idesc_mx(M, N, fmt_a, fmt_b);
}

int64_t gemm_mxf8_sf_offset(int64_t row, int64_t k_block, int64_t K)
{
    if (row < 0 || k_block < 0 || K < 0 || K % 32 != 0 || k_block >= K / 32) return -1;
    return static_cast<int64_t>(gf16::mx_sf_offset(static_cast<uint64_t>(row),
                                                   static_cast<uint32_t>(k_block),
                                                   gf16::mx_k_groups(static_cast<uint32_t>(K / 32))));
}

uint64_t gemm_mxf8_sf_desc(uint32_t smem_addr) { return gf16::make_sf_desc(smem_addr); }

int gemm_mxf8_get_variant_info(int variant, gemm_f16_variant_info* o)
{
    if (!o) return GEMM_F16_ERR_INVALID_ARG;
    switch (variant) {
    case GEMM_MXF8_VARIANT_128x128:
        *o = {1, 128, 128, 128, 5, (int)MxCta::THREADS, (int)MxCta::SMEM_ALLOC,
              (int)MxCta::TMEM_COLS, (int)MxCta::STAGE_TX, 1};
        return GEMM_F16_OK;
    case GEMM_MXF8_VARIANT_PAIR_256x128:
        *o = {2, 256, 128, 128, 7, (int)MxPair::THREADS, (int)MxPair::SMEM_ALLOC,
              (int)MxPair::TMEM_COLS, (int)MxPair::STAGE_TX, 1};
        return GEMM_F16_OK;
    case GEMM_MXF8_VARIANT_PAIR_256x192:
        *o = {2, 256, 192, 128, 6, (int)MxPair192::THREADS, (int)MxPair192::SMEM_ALLOC,
              (int)MxPair192::TMEM_COLS, (int)MxPair192::STAGE_TX, 1};
        return GEMM_F16_OK;
    case GEMM_MXF8_VARIANT_PAIR_256x256:
        *o = {2, 256, 256, 128, 6, (int)MxPair256::THREADS, (int)MxPair256::SMEM_ALLOC,
              (int)MxPair256::TMEM_COLS, (int)MxPair256::STAGE_TX, 1};
        return GEMM_F16_OK;
    default:
        return GEMM_F16_ERR_INVALID_ARG;
    }
}

void gemm_f16_ring_pos(uint32_t it, uint32_t stages, uint32_t* stage, uint32_t* parity)
{
    const gf16::RingPos p = gf16::ring_pos(it, stages);
    if (stage) *stage = p.stage;
    if (parity) *parity = p.parity;
}

}  // extern "C"
