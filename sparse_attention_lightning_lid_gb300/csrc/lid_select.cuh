// lid_select.cuh -- exact top-k building blocks on 64-bit composite keys.
//
// A key packs (score, index) so that one unsigned comparison orders by score
// descending and then index ascending:
//   key = ord(score) << 32 | ~index
// where ord maps IEEE binary32 bits to an unsigned integer of the same order
// (negative values: all bits flipped; non-negative: sign bit set), after
// folding -0 onto +0 so both compare equal. Every real key is non-zero
// (~index >= 2^31 for index < 2^31), so 0 marks an empty slot.
//
// The selection is a most-significant-digit radix select (8-bit digits): a
// histogram of the current digit among keys that share the prefix found so
// far locates the digit of the k-th largest key; it stops as soon as the
// whole bucket is taken. Keys are unique, so after at most eight passes the
// k largest keys are exactly those whose masked high bits are >= the prefix.
#pragma once

#include <stdint.h>

#include "lid_ptx.cuh"

namespace lid {

__device__ __forceinline__ uint32_t ord_f32(float f) {
    uint32_t u = __float_as_uint(f);
    if (u == 0x80000000u) u = 0u;  // -0 -> +0
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__device__ __forceinline__ float unord_f32(uint32_t o) {
    const uint32_t u = (o & 0x80000000u) ? (o & 0x7FFFFFFFu) : ~o;
    return __uint_as_float(u);
}

__device__ __forceinline__ uint64_t make_key(float score, uint32_t idx) {
    return (static_cast<uint64_t>(ord_f32(score)) << 32) | static_cast<uint64_t>(~idx);
}

__device__ __forceinline__ void decode_key(uint64_t key, int32_t &idx, float &score) {
    if (key == 0) {
        idx = -1;
        score = __uint_as_float(0xFF800000u);  // -inf
    } else {
        idx = static_cast<int32_t>(~static_cast<uint32_t>(key));
        score = unord_f32(static_cast<uint32_t>(key >> 32));
    }
}

// Scratch a group of NW warps shares while cutting with DB-bit digits.
template <int DB, int NW>
struct CutScratch {
    int hist[3][1 << DB];
    unsigned long long wlo[NW];
    unsigned long long whi[NW];
    unsigned long long wkept[NW];  // separate from wlo: a following call may refill wlo early
};

// Scratch of the bucket sort (8-bit digits) for a group of NW warps.
template <int NW>
struct SortScratch {
    int hist[256];
    int fill[256];
    unsigned long long wlo[NW];  // per warp: smallest / largest finite-score key
    unsigned long long whi[NW];
    unsigned long long wall[2];  // folded smallest / largest
};

// Append `key` to buf (counter *cnt) for lanes where `ins` is set, one
// shared-memory atomic per warp. All 32 lanes must call it. Returns the
// counter value just after this warp's append (same on every lane).
__device__ __forceinline__ int warp_append(uint64_t *buf, int *cnt, uint64_t key, bool ins, int lane) {
    const unsigned bal = __ballot_sync(0xFFFFFFFFu, ins);
    if (bal == 0u) return 0;
    const int leader = __ffs(bal) - 1;
    int base = 0;
    if (lane == leader) base = atomicAdd(cnt, __popc(bal));
    base = __shfl_sync(0xFFFFFFFFu, base, leader);
    if (ins) buf[base + __popc(bal & ((1u << lane) - 1u))] = key;
    return base + __popc(bal);
}

__device__ __forceinline__ unsigned long long warp_min_u64(unsigned long long v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const unsigned long long x = __shfl_xor_sync(0xFFFFFFFFu, v, o);
        v = x < v ? x : v;
    }
    return v;
}

__device__ __forceinline__ unsigned long long warp_max_u64(unsigned long long v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const unsigned long long x = __shfl_xor_sync(0xFFFFFFFFu, v, o);
        v = x > v ? x : v;
    }
    return v;
}

// Sorts one value per lane descending across the warp (bitonic network):
// lane i returns the (i+1)-th largest. All 32 lanes must call it.
__device__ __forceinline__ unsigned long long warp_sort_desc_u64(unsigned long long v, int lane) {
#pragma unroll
    for (int k = 2; k <= 32; k <<= 1) {
#pragma unroll
        for (int j = k >> 1; j > 0; j >>= 1) {
            const unsigned long long o = __shfl_xor_sync(0xFFFFFFFFu, v, j);
            // blocks of k lanes alternate direction; the last (k = 32) is descending
            const bool take_max = ((lane & j) == 0) == ((lane & k) == 0);
            v = take_max ? (o > v ? o : v) : (o < v ? o : v);
        }
    }
    return v;
}

// DB-bit digit of `key` whose lowest bit is bit `shift` (shift may be
// negative near the end: the missing low bits read as zero).
template <int DB>
__device__ __forceinline__ int key_digit(uint64_t key, int shift) {
    return static_cast<int>((shift >= 0 ? (key >> shift) : (key << (-shift))) & ((1u << DB) - 1u));
}

template <int DB>
__device__ __forceinline__ uint64_t digit_mask(int shift) {
    constexpr uint64_t M = (1ull << DB) - 1ull;
    return shift >= 0 ? (M << shift) : (M >> (-shift));
}

__device__ __forceinline__ uint64_t digit_bits(int d, int shift) {
    return shift >= 0 ? (static_cast<uint64_t>(d) << shift) : (static_cast<uint64_t>(d) >> (-shift));
}

// Exclusive prefix sum of v over the T threads (tid < T, T a multiple of 32,
// at most 1024) on named barrier `bar`, without atomics: a warp scan, then the
// warp totals through `wtot` (32 ints of shared memory). Returns the sum over
// threads below tid; *total gets the sum over all. Ends with a barrier, after
// which wtot may be reused.
template <int T>
__device__ __forceinline__ int block_excl_scan(int v, int tid, int bar, int *wtot, int *total) {
    constexpr int NW = T / 32;
    const int lane = tid & 31, warp = tid >> 5;
    int incl = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int x = __shfl_up_sync(0xFFFFFFFFu, incl, o);
        if (lane >= o) incl += x;
    }
    if (lane == 31) wtot[warp] = incl;
    named_bar(bar, T);
    int base = 0, all = 0;
    for (int w = 0; w < NW; ++w) {
        const int x = wtot[w];
        base += w < warp ? x : 0;
        all += x;
    }
    named_bar(bar, T);
    *total = all;
    return base + incl - v;
}

// Exactly the c-th largest (1-based) of the values a warp holds, V per lane
// (0 = no value; ties count separately), by a most-significant-bit-first
// radix select on ballots: returns 0 when fewer than c values are non-zero.
// Uniform across the warp; all 32 lanes must call it.
template <int V>
__device__ __forceinline__ uint32_t warp_kth_largest(const uint32_t (&o)[V], int c) {
    uint32_t prefix = 0u, mask = 0u;
    int remaining = c;
#pragma unroll 1
    for (int b = 31; b >= 0; --b) {
        const uint32_t bit = 1u << b;
        int cnt = 0;
#pragma unroll
        for (int k = 0; k < V; ++k) cnt += __popc(__ballot_sync(0xFFFFFFFFu, (o[k] & mask) == prefix && (o[k] & bit)));
        if (cnt >= remaining) prefix |= bit;
        else remaining -= cnt;
        mask |= bit;
    }
    // prefix is the c-th largest value if at least c values exist, else the
    // search ran down to 0 with remaining > 0
    int nz = 0;
#pragma unroll
    for (int k = 0; k < V; ++k) nz += __popc(__ballot_sync(0xFFFFFFFFu, o[k] != 0u));
    return nz >= c ? prefix : 0u;
}

// Smallest and largest key of buf[0, n), uniform across the group of NW
// warps. Ends with a barrier; before it, also zeroes zero[0, nzero) and, if
// given, *count.
template <int NW>
__device__ __forceinline__ void group_minmax(const uint64_t *buf, int n, int tid, int bar, unsigned long long *wlo,
                                             unsigned long long *whi, int *zero, int nzero, uint64_t &lo,
                                             uint64_t &hi, int *count = nullptr) {
    constexpr int T = 32 * NW;
    const int lane = tid & 31, warp = tid >> 5;
    unsigned long long l = ~0ull, h = 0ull;
    for (int i = tid; i < n; i += T) {
        const unsigned long long key = buf[i];
        l = key < l ? key : l;
        h = key > h ? key : h;
    }
    l = warp_min_u64(l);
    h = warp_max_u64(h);
    if (lane == 0) {
        wlo[warp] = l;
        whi[warp] = h;
    }
    for (int i = tid; i < nzero; i += T) zero[i] = 0;
    if (tid == 0 && count != nullptr) *count = 0;
    named_bar(bar, T);
    lo = ~0ull;
    hi = 0ull;
#pragma unroll
    for (int w = 0; w < NW; ++w) {
        lo = wlo[w] < lo ? wlo[w] : lo;
        hi = whi[w] > hi ? whi[w] : hi;
    }
}

// Every warp scans the histogram the same way, so the result is uniform
// without another barrier: the digit d holding the key of rank `remaining`
// (counted from the largest), the count in higher digits, and the count in d.
template <int DB>
__device__ __forceinline__ void scan_digit(const int *hist, int remaining, int lane, int &d, int &above,
                                           int &inbin) {
    constexpr int B = 1 << DB;
    constexpr int PL = B >= 32 ? B / 32 : 1;  // bins per lane (lanes >= B own none)
    int c[PL];
    int tot = 0;
#pragma unroll
    for (int j = 0; j < PL; ++j) {
        const int bin = PL * lane + j;
        c[j] = bin < B ? hist[bin] : 0;
        tot += c[j];
    }
    int incl = tot;  // inclusive suffix sum over lanes >= lane (higher digits)
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int v = __shfl_down_sync(0xFFFFFFFFu, incl, o);
        if (lane + o < 32) incl += v;
    }
    const int above_lane = incl - tot;
    int res = -1, r_above = 0, r_in = 0;
    if (above_lane < remaining && remaining <= incl) {
        int a = above_lane;
#pragma unroll
        for (int j = PL - 1; j >= 0; --j) {
            if (res < 0 && a + c[j] >= remaining) {
                res = PL * lane + j;
                r_above = a;
                r_in = c[j];
            }
            a += c[j];
        }
    }
    const unsigned who = __ballot_sync(0xFFFFFFFFu, res >= 0);
    const int src = who ? __ffs(who) - 1 : 0;
    d = __shfl_sync(0xFFFFFFFFu, res, src);
    above = __shfl_sync(0xFFFFFFFFu, r_above, src);
    inbin = __shfl_sync(0xFFFFFFFFu, r_in, src);
}

// Cut buf[0, n) of unique keys (n > k) down to the keys at or above a
// threshold that keeps at least k of them. exact = true keeps exactly the k
// largest; exact = false stops as soon as at most k + slack keys remain (the
// cheap cut used while streaming). Run by the NW warps of a group (named
// barrier `bar`, tid in [0, 32 NW); up to 32 NW R keys are compacted through
// registers, more in barrier-separated rounds); the kept keys end up in
// buf[0, kept) unordered and *count = kept. Returns kept; *min_kept is the
// smallest kept key (both uniform across the group).
//
// Most-significant-digit radix select on DB-bit digits, starting just below
// the bits all keys share (from their minimum and maximum), so the first
// digit already spreads the keys over many bins and the histogram's
// shared-memory atomics rarely collide.
template <int R, int DB, int NW>
__device__ __noinline__ int group_cut(uint64_t *buf, int *count, int n, int k, int slack, bool exact, int tid, int bar,
                         CutScratch<DB, NW> *sc, uint64_t *min_kept) {
    constexpr int T = 32 * NW;
    constexpr int B = 1 << DB;
    const int lane = tid & 31, warp = tid >> 5;
    uint64_t lo, hi;
    unsigned long long mymin = ~0ull;
    int kept = n;
    if (n <= T * R) {
        // every key in registers: read once for the min / max, the digit passes
        // and the compaction
        uint64_t v[R];
        unsigned long long l = ~0ull, h = 0ull;
#pragma unroll
        for (int r = 0; r < R; ++r) {
            const int i = r * T + tid;
            v[r] = i < n ? buf[i] : 0ull;
            if (i < n) {
                l = v[r] < l ? v[r] : l;
                h = v[r] > h ? v[r] : h;
            }
        }
        l = warp_min_u64(l);
        h = warp_max_u64(h);
        if (lane == 0) {
            sc->wlo[warp] = l;
            sc->whi[warp] = h;
        }
        for (int i = tid; i < B; i += T) sc->hist[0][i] = 0;
        named_bar(bar, T);
        lo = ~0ull;
        hi = 0ull;
#pragma unroll
        for (int w = 0; w < NW; ++w) {
            lo = sc->wlo[w] < lo ? sc->wlo[w] : lo;
            hi = sc->whi[w] > hi ? sc->whi[w] : hi;
        }
        const uint64_t diff = lo ^ hi;  // non-zero: keys are unique and n >= 2
        const int hb = 63 - __clzll(static_cast<long long>(diff));
        uint64_t pmask = hb >= 63 ? 0ull : ~((2ull << hb) - 1ull);
        uint64_t prefix = lo & pmask;
        int remaining = k;
        for (int shift = hb - (DB - 1), pass = 0;; shift -= DB, ++pass) {
            int *hist = sc->hist[pass % 3];
            int *next = sc->hist[(pass + 1) % 3];  // last read two passes ago
            for (int i = tid; i < B; i += T) next[i] = 0;
#pragma unroll
            for (int r = 0; r < R; ++r) {
                const int i = r * T + tid;
                if (i < n && (v[r] & pmask) == prefix) atomicAdd(&hist[key_digit<DB>(v[r], shift)], 1);
            }
            named_bar(bar, T);
            int d, above, inbin;
            scan_digit<DB>(hist, remaining, lane, d, above, inbin);
            prefix |= digit_bits(d, shift);
            pmask |= digit_mask<DB>(shift);
            remaining -= above;
            kept = (k - remaining) + inbin;  // keys at or above this prefix
            if (inbin == remaining || shift <= 0) break;
            if (!exact && kept <= k + slack) break;
        }
        // positions from a scan over the group (no atomics on the count); every
        // key was read before the first barrier above, so the writes may follow
        int mine = 0;
#pragma unroll
        for (int r = 0; r < R; ++r) mine += (r * T + tid < n && (v[r] & pmask) >= prefix) ? 1 : 0;
        int incl = mine;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int x = __shfl_up_sync(0xFFFFFFFFu, incl, o);
            if (lane >= o) incl += x;
        }
        if (lane == 31) sc->wkept[warp] = static_cast<unsigned long long>(incl);
        named_bar(bar, T);
        int pos = incl - mine, total = 0;
#pragma unroll
        for (int w = 0; w < NW; ++w) {
            const int x = static_cast<int>(sc->wkept[w]);
            pos += w < warp ? x : 0;
            total += x;
        }
#pragma unroll
        for (int r = 0; r < R; ++r) {
            if (r * T + tid < n && (v[r] & pmask) >= prefix) {
                buf[pos++] = v[r];
                if (v[r] < mymin) mymin = v[r];
            }
        }
        if (tid == 0) *count = total;
        named_bar(bar, T);  // every thread has read wkept before it is reused below
    } else {
        group_minmax<NW>(buf, n, tid, bar, sc->wlo, sc->whi, sc->hist[0], B, lo, hi, count);
        const uint64_t diff = lo ^ hi;  // non-zero: keys are unique and n >= 2
        const int hb = 63 - __clzll(static_cast<long long>(diff));
        uint64_t pmask = hb >= 63 ? 0ull : ~((2ull << hb) - 1ull);
        uint64_t prefix = lo & pmask;
        int remaining = k;
        for (int shift = hb - (DB - 1), pass = 0;; shift -= DB, ++pass) {
            int *hist = sc->hist[pass % 3];
            int *next = sc->hist[(pass + 1) % 3];  // last read two passes ago
            for (int i = tid; i < B; i += T) next[i] = 0;
            for (int base = 0; base < n; base += T) {
                const int i = base + tid;
                if (i < n) {
                    const uint64_t key = buf[i];
                    if ((key & pmask) == prefix) atomicAdd(&hist[key_digit<DB>(key, shift)], 1);
                }
            }
            named_bar(bar, T);
            int d, above, inbin;
            scan_digit<DB>(hist, remaining, lane, d, above, inbin);
            prefix |= digit_bits(d, shift);
            pmask |= digit_mask<DB>(shift);
            remaining -= above;
            kept = (k - remaining) + inbin;  // keys at or above this prefix
            if (inbin == remaining || shift <= 0) break;
            if (!exact && kept <= k + slack) break;
        }
        // compaction in rounds: round r reads buf[rT, rT + T) and writes kept
        // keys below (r + 1) T, so a barrier between its reads and writes suffices
        for (int base = 0; base < n; base += T) {
            const int i = base + tid;
            const uint64_t key = i < n ? buf[i] : 0ull;
            const bool keep = (i < n) && ((key & pmask) >= prefix);
            named_bar(bar, T);
            warp_append(buf, count, key, keep, lane);
            if (keep && key < mymin) mymin = key;
        }
    }
    mymin = warp_min_u64(mymin);
    if (lane == 0) sc->wkept[warp] = mymin;
    named_bar(bar, T);
    unsigned long long mk = ~0ull;
#pragma unroll
    for (int w = 0; w < NW; ++w) mk = sc->wkept[w] < mk ? sc->wkept[w] : mk;
    *min_kept = mk;
    return kept;
}

// Bucket of a key for the sort: linear in the score between the smallest
// and largest finite score of the keys, so the top-k of a smooth score
// distribution spreads evenly (bits-based digits would crowd keys of one
// binade into a few buckets). Non-decreasing in the key; -inf goes to 0.
__device__ __forceinline__ int value_bucket(uint64_t key, float s_lo, float scale) {
    const float s = unord_f32(static_cast<uint32_t>(key >> 32));
    if (!(s > s_lo)) return 0;  // s_lo itself, and -inf
    const float b = (s - s_lo) * scale;
    return b >= 255.f ? 255 : static_cast<int>(b);
}

// Sort buf[0, n) (unique keys, n <= 32 NW R) descending, in place, using
// tmp[0, n) as scratch: a counting sort on value_bucket(), then each key's
// place inside its bucket is its count of larger keys in the bucket (a
// bucket crowded by equal scores costs O(bucket^2)). Ends with a barrier.
template <int R, int NW>
__device__ __noinline__ void group_sort_desc(uint64_t *buf, uint64_t *tmp, int n, int tid, int bar, SortScratch<NW> *sc) {
    constexpr int T = 32 * NW;
    if (n <= 1) {
        named_bar(bar, T);
        return;
    }
    const int lane = tid & 31, warp = tid >> 5;
    // smallest and largest finite score (keys below kFinite hold -inf); warp 0
    // folds the per-warp values and publishes them
    constexpr uint64_t kFinite = 0x00800000ull << 32;
    constexpr uint64_t kPosInf = static_cast<uint64_t>(0xFF800000u) << 32;  // ord(+inf) << 32
    unsigned long long l = ~0ull, h = 0ull;
    uint64_t v[R];
#pragma unroll
    for (int r = 0; r < R; ++r) {
        const int i = r * T + tid;
        v[r] = i < n ? buf[i] : 0ull;
        if (i < n && v[r] >= kFinite && v[r] < kPosInf) {
            l = v[r] < l ? v[r] : l;
            h = v[r] > h ? v[r] : h;
        }
    }
    l = warp_min_u64(l);
    h = warp_max_u64(h);
    if (lane == 0) {
        sc->wlo[warp] = l;
        sc->whi[warp] = h;
    }
    for (int i = tid; i < 256; i += T) sc->hist[i] = 0;
    named_bar(bar, T);
    if (warp == 0) {
        unsigned long long lo = lane < NW ? sc->wlo[lane] : ~0ull;
        unsigned long long hi = lane < NW ? sc->whi[lane] : 0ull;
        lo = warp_min_u64(lo);
        hi = warp_max_u64(hi);
        if (lane == 0) {
            sc->wall[0] = lo;
            sc->wall[1] = hi;
        }
    }
    named_bar(bar, T);
    const unsigned long long lo = sc->wall[0], hi = sc->wall[1];
    float s_lo = 0.f, scale = 0.f;
    if (lo != ~0ull && hi != 0ull) {
        s_lo = unord_f32(static_cast<uint32_t>(lo >> 32));
        const float s_hi = unord_f32(static_cast<uint32_t>(hi >> 32));
        if (s_hi > s_lo) scale = 255.f / (s_hi - s_lo);
        if (!(scale < __uint_as_float(0x7F800000u))) scale = 0.f;  // range too small to divide
    }
    int hb = 0;
    if (scale == 0.f) {
        // no score spread (ties, or no finite scores): bucket on the key bits
        // below the bits all keys share instead (rare; one more reduction)
        unsigned long long la = ~0ull, ha = 0ull;
#pragma unroll
        for (int r = 0; r < R; ++r) {
            if (r * T + tid < n) {
                la = v[r] < la ? v[r] : la;
                ha = v[r] > ha ? v[r] : ha;
            }
        }
        la = warp_min_u64(la);
        ha = warp_max_u64(ha);
        if (lane == 0) sc->wlo[warp] = la ^ ha;  // spread of this warp's keys
        named_bar(bar, T);
        unsigned long long spread = 0ull;
#pragma unroll
        for (int w = 0; w < NW; ++w) spread |= sc->wlo[w];
        hb = spread ? 63 - __clzll(static_cast<long long>(spread)) : 0;
    }
    int dg[R];
#pragma unroll
    for (int r = 0; r < R; ++r) {
        if (r * T + tid < n) dg[r] = scale > 0.f ? value_bucket(v[r], s_lo, scale) : key_digit<8>(v[r], hb - 7);
        else dg[r] = -1;
        if (dg[r] >= 0) atomicAdd(&sc->hist[dg[r]], 1);
    }
    named_bar(bar, T);
    // bucket starts in descending bucket order; lane l of warp 0 owns buckets 8l..8l+7
    if (tid < 32) {
        int c[8], tot = 0;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            c[j] = sc->hist[8 * lane + j];
            tot += c[j];
        }
        int incl = tot;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int x = __shfl_down_sync(0xFFFFFFFFu, incl, o);
            if (lane + o < 32) incl += x;
        }
        int start = incl - tot;  // keys in higher buckets
#pragma unroll
        for (int j = 7; j >= 0; --j) {
            sc->fill[8 * lane + j] = start;  // running slot of bucket 8l+j
            start += c[j];
        }
    }
    named_bar(bar, T);
#pragma unroll
    for (int r = 0; r < R; ++r) {
        if (dg[r] >= 0) tmp[atomicAdd(&sc->fill[dg[r]], 1)] = v[r];
    }
    named_bar(bar, T);
    // place: bucket start (fill now points one past the bucket) + larger keys in the bucket
#pragma unroll
    for (int r = 0; r < R; ++r) {
        if (dg[r] >= 0) {
            const int size = sc->hist[dg[r]];
            const int start = sc->fill[dg[r]] - size;
            int rank = 0, j = start;
            for (; j + 4 <= start + size; j += 4)  // four independent loads per step
                rank += (tmp[j] > v[r]) + (tmp[j + 1] > v[r]) + (tmp[j + 2] > v[r]) + (tmp[j + 3] > v[r]);
            for (; j < start + size; ++j) rank += tmp[j] > v[r];
            buf[start + rank] = v[r];
        }
    }
    named_bar(bar, T);
}

}  // namespace lid
