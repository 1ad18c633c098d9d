// The packed-sequence offsets' contract of the Gated Delta Net prefill, shared by the device
// kernels that enforce it and the host copy the tests replay (page "TIRx" (zixuwang.me), section
// "用状态递推解释 GDN", packed input: a sequence's replay never crosses its cu_seqlens boundary).
//
// cu_seqlens[0 .. n_seqs] must start at 0, end at total_tokens and never decrease; then every
// sequence's tokens lie inside [0, total_tokens) and the sequences do not overlap.  A call whose
// offsets break this is refused on the device: its status word gets kGdnStatusBadOffsets, every
// sequence is treated as empty (no token is read or written; states pass through), and
// gdn_check_status reports GDN_ERR_INVALID_ARG.
#ifndef GDN_OFFSETS_H
#define GDN_OFFSETS_H

#include <stdint.h>

#if defined(__CUDACC__)
#define GDN_HD __host__ __device__ __forceinline__
#else
#define GDN_HD inline
#endif

namespace gdn {

// Bits of a call's status word (in the workspace; cleared by the call's first kernel).
constexpr uint32_t kStatusTimeout = 1u;      // a scan CTA gave up a bounded wait for its loads
constexpr uint32_t kStatusBadOffsets = 2u;   // cu_seqlens broke its contract

// One neighbouring pair (cu[i], cu[i + 1]).
GDN_HD bool offsets_pair_ok(int32_t lo, int32_t hi) { return lo <= hi; }

// The two ends (cu[0], cu[n_seqs]).
GDN_HD bool offsets_ends_ok(int32_t first, int32_t last, int64_t total_tokens)
{
    return first == 0 && static_cast<int64_t>(last) == total_tokens;
}

// One sequence, whose kernels number the chunks from total_tokens alone: its two offsets must be
// exactly [0, total_tokens].
GDN_HD bool offsets_single_ok(int32_t first, int32_t last, int64_t total_tokens)
{
    return offsets_ends_ok(first, last, total_tokens);
}

}  // namespace gdn

#endif  // GDN_OFFSETS_H
