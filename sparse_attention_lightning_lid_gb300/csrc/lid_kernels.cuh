// lid_kernels.cuh -- the lightning-indexer scoring + streaming top-k kernel
// (with, in its one-launch form, the merge of the key splits) and the
// two-launch split merge kernel, sm_103a.
//
// Per CTA: one group of QG queries (QG*H rows of q, the MMA's N) and one
// contiguous range of 128-key tiles (a split; with per-row visible ranges,
// a split of the tiles the group's ranges touch). Warp roles:
//   warp 0      TMA producer: q once, then each K tile into a ring of stages
//   warp 1      allocates tensor memory and issues tcgen05.mma: S = K_tile . Q^T,
//               keys on M (128 TMEM lanes), query x head on N, into one of
//               `acc_stages` fp32 accumulators in TMEM
//   warps 2..17 epilogue, in four groups of four warps (one warp per TMEM lane
//               quarter); group g owns a quarter of the queries. Each thread
//               owns one key (its TMEM lane) and, for each of its group's
//               queries, sums w[t,h] * relu(S) over that query's H columns in
//               registers, adds mask[t,s], and appends the key to the query's
//               candidate buffer if it beats the query's running threshold. A
//               buffer that could overflow on the next tile is cut back (radix
//               prune) to a little over top_k keys, which raises the threshold.
//               Groups synchronise only among themselves, so their cuts and
//               final sorts run side by side. With one query per CTA the
//               groups instead take tiles in turn (when no cut can be
//               needed), or some stream while the others run the one-launch
//               path's certificate steps.
// Nothing of size n_q x n_kv is written: scores exist only in TMEM/registers.
#pragma once

#include <cuda_fp16.h>
#include <stdint.h>

#include "lid_ptx.cuh"
#include "lid_select.cuh"

namespace lid {

constexpr int kBM = 128;        // keys per tile (MMA M, TMEM lanes)
constexpr int kMaxQG = 32;      // queries per CTA at most (H = 8)
constexpr int kMaxKStages = 8;
constexpr int kMaxAccStages = 4;
constexpr int kEpiBar = 1;      // named barrier of all epilogue warps (2..5: one per group)
constexpr int kEPG = 4;         // epilogue groups = epilogue warps per TMEM lane quarter
constexpr int kEpiThreads = 128 * kEPG;
constexpr int kScoreThreads = 64 + kEpiThreads;  // + TMA warp + MMA warp
constexpr int kMaxCap = 4096;   // candidate keys per query
constexpr int kMaxCapRanges = 8192;  // ... for one query per CTA with visible ranges (see the planner)
constexpr int kSortMax = 2048;  // keys a final sort takes at once (more are first cut to top_k)
constexpr int kCutDB = 6;       // digit bits of the streaming cuts
constexpr int kSortScratchBytes = (static_cast<int>(sizeof(SortScratch<16>)) + 63) & ~63;
constexpr int kCutScratchBytes = (static_cast<int>(sizeof(CutScratch<8, 16>)) + 63) & ~63;
// final-phase scratch one sorter needs (counters + kSortMax keys)
constexpr int kFinalScratchBytes = kSortScratchBytes + kCutScratchBytes + kSortMax * 8;

// One-launch split path: sizes of its global and shared scratch.
constexpr int kFusedLevels = 8;                    // certificates per CTA and query: ranks 1, 2, 4, ..., 128
constexpr int kFusedRounds = 8;                    // histogram rounds that can tighten a bound
constexpr int kFusedAttempts = kFusedRounds + 1;   // candidate gathers per query at most
constexpr int kFusedCapMax = 4096;                 // candidates per query gathered for the ranking

struct ScoreParams {
    const uint16_t *mask;  // [n_q][n_kv] f16 bits or null
    const int32_t *row_lo, *row_hi;  // or [n_q] visible key ranges [lo, hi) (keys outside score -inf)
    const float *w;        // [n_q][H]
    // 8-bit operands (esize 1): q and k are E4M3 codes, an element's value is
    // its row's scale times the code's value; null (and esize 2) for 16-bit
    const float *q_scale;  // [n_q][H]
    const float *k_scale;  // [n_kv]
    int esize;             // bytes per q / k element: 2 (bf16, f16) or 1 (E4M3, D = 128 only)
    int32_t *out_idx;      // [n_q][top_k] (splits == 1)
    float *out_score;
    uint64_t *part;        // [n_q][splits][top_k] sorted keys (splits > 1)
    long long n_q, n_kv;
    int D, QG, N, top_k, P;  // P = top_k rounded up to a power of two
    int n_groups, splits, tiles_per_split, n_tiles;
    int kstages, acc_stages, cap, tmem_cols;
    uint32_t idesc;
    long long wait_limit;  // cycles a wait may last before the CTA aborts
    int fault;             // test hooks: 2, the epilogue waits on a barrier nothing completes;
                           // 3, the first group barrier of the one-launch path waits for one CTA too many
    // one-launch split path (all CTAs of a query group resident together)
    unsigned *f_bar;       // [n_groups] arrival counters, zero when the launch starts
    unsigned *f_done;      // [n_groups] CTAs finished; non-null: the last CTA of a group re-zeroes
                           // both counters on its way out (a slot that stays clean between launches)
    int *f_count;          // [n_q][kFusedAttempts] candidate counts
    int *f_hist;           // [kFusedRounds][n_q][256] digit histograms
    uint64_t *f_stats;     // [n_q][kFusedLevels][splits] certificates
    uint64_t *f_cand;      // [n_q][f_cap] gathered candidates
    int f_cap;
    int tilepar;           // (one query per CTA, no cut possible) 2 or 4: that many epilogue groups take tiles in turn
    int f_early;           // 1: steps A-B run on the idle epilogue warps while group 0 streams
    int f_pub;             // (early) tiles streamed before the certificates are published
    uint64_t *f_reg;       // (early) [n_q][splits][f_regcap + 1]: per split a count, then its keys >= the
                           // bound (null: gather through f_cand only)
    int f_regcap;          // keys a split's region holds
    int side_bulk;         // (single-query kernel) bit 0: the mask rows, bit 1: the key scales may be
                           // fetched with 16-byte aligned bulk copies
    // (split lists, splits > 1) [n_q], zero when the launch starts: per query the largest key v
    // that some split has certified, i.e. it holds at least top_k keys >= v, so the query's
    // top_k-th key is >= v and every split may drop the keys below v; null: not used
    unsigned long long *qbound;
};

struct Misc {
    uint64_t k_full[kMaxKStages];
    uint64_t k_empty[kMaxKStages];
    uint64_t acc_full[kMaxAccStages];
    uint64_t acc_empty[kMaxAccStages];
    uint64_t q_full;
    uint64_t mma_done;  // all MMAs of the CTA finished (before TMEM is freed)
    uint64_t never;     // a barrier nothing arrives at (the fault-injection test)
    int cnt[kMaxQG];
    int qlo[kMaxQG], qhi[kMaxQG];  // (ranges) each query's visible keys, clamped to [0, n_kv]
    int tile0, ntl;                // this CTA's tiles
    CutScratch<kCutDB, 4> cut[kEPG];
    uint32_t tmem_base;
    int abort_flag;
    unsigned long long live_bound;  // (early) the certified bound once steps A-B are done, else 0
};

struct SmemLayout {
    uint32_t stage_bytes, k_off, q_off, w_off, buf_off, misc_off, early_off, total;
};

// Offsets from a 1024-byte aligned base; `total` includes the alignment slack.
// early_bytes: scratch of the one-launch path's early steps (0: none).
__host__ __device__ inline SmemLayout smem_layout(int D, int N, int QG, int H, int kstages, int cap,
                                                  uint32_t early_bytes = 0) {
    SmemLayout L;
    L.stage_bytes = static_cast<uint32_t>(kBM * D * 2);
    L.k_off = 0;
    L.q_off = L.k_off + L.stage_bytes * kstages;
    L.w_off = L.q_off + static_cast<uint32_t>(N * D * 2);
    L.buf_off = L.w_off + ((static_cast<uint32_t>(QG * H * 4) + 15u) & ~15u);
    L.misc_off = L.buf_off + static_cast<uint32_t>(QG) * static_cast<uint32_t>(cap) * 8u;
    L.early_off = L.misc_off + ((static_cast<uint32_t>(sizeof(Misc)) + 127u) & ~127u);
    L.total = L.early_off + early_bytes + 1024u;
    return L;
}

// Epilogue groups that own at least one query, and queries per group.
__host__ __device__ inline int queries_per_group(int QG) { return (QG + kEPG - 1) / kEPG; }
__host__ __device__ inline int active_groups(int QG) {
    const int qpg = queries_per_group(QG);
    return (QG + qpg - 1) / qpg;
}

// Bytes of K-stage shared memory each final-phase sorter may use as scratch
// (the stages are idle once the last tile has been consumed).
__host__ __device__ inline uint32_t final_scratch_bytes(int QG, uint32_t kstage_total) {
    return QG == 1 ? kstage_total : kstage_total / static_cast<uint32_t>(active_groups(QG));
}

constexpr uint16_t kF16NegInf = 0xFC00u;  // f16 bits of -inf

__device__ __forceinline__ float f16_bits_to_float(uint16_t b) {
    return __half2float(__ushort_as_half(b));
}

// Sort the n candidate keys of row t and write the top_k: the final output
// row (splits == 1) or this split's sorted list. More than kSortMax keys are
// first cut to exactly top_k. `scratch` holds the cut's and the sort's
// counters followed by kSortMax keys of temporary space.
template <int NW>
__device__ __noinline__ void finish_row(uint64_t *b, int *cnt, uint8_t *scratch, const ScoreParams &p, long long t, int split,
                           int tid, int bar) {
    constexpr int T = 32 * NW;
    SortScratch<NW> *ss = reinterpret_cast<SortScratch<NW> *>(scratch);
    CutScratch<8, NW> *cs = reinterpret_cast<CutScratch<8, NW> *>(scratch + kSortScratchBytes);
    uint64_t *tmp = reinterpret_cast<uint64_t *>(scratch + kSortScratchBytes + kCutScratchBytes);
    int n = *cnt;
    if (n > kSortMax) {
        uint64_t mk;
        group_cut<kSortMax / T, 8, NW>(b, cnt, n, p.top_k, 0, true, tid, bar, cs, &mk);
        n = p.top_k;
    }
    group_sort_desc<kSortMax / T, NW>(b, tmp, n, tid, bar, ss);
    // this split's top_k-th key: the split holds top_k keys >= it (see ScoreParams::qbound)
    if (p.qbound != nullptr && n >= p.top_k && tid == 0)
        atomicMax(p.qbound + t, static_cast<unsigned long long>(b[p.top_k - 1]));
    if (p.splits == 1) {
        for (int j = tid; j < p.top_k; j += T) {
            int32_t idx;
            float sc;
            decode_key(j < n ? b[j] : 0ull, idx, sc);
            p.out_idx[t * p.top_k + j] = idx;
            p.out_score[t * p.top_k + j] = sc;
        }
    } else {
        uint64_t *dst = p.part + (t * p.splits + split) * static_cast<long long>(p.top_k);
        for (int j = tid; j < p.top_k; j += T) dst[j] = j < n ? b[j] : 0ull;
    }
    named_bar(bar, T);
}

// ------------------------------------------------- one-launch split path
// When every CTA of a query group fits on the GPU at once (a cooperative
// launch), the per-split top-k lists and the separate merge are replaced by
// two group barriers inside the scoring kernel. Each step handles all the
// group's queries together, so they share the barriers.
//
//  A. Certificates. A CTA's keys of query t fall into 128 rows (index mod
//     128, one epilogue thread each). If u_r is the r-th largest row maximum,
//     the CTA has at least r keys >= u_r. The row maxima are sorted within
//     each TMEM lane quarter (one warp each), ranked across the four sorted
//     quarters by binary search, and u_r is published for r = 1, 2, ..., 128.
//  B. Bound. If c = ceil(top_k / r) CTAs each have r keys >= v, at least
//     top_k keys are >= v; so the c-th largest published u_r (over the
//     splits) is a lower bound on the query's top_k-th key, and so is the
//     lower edge of a histogram bin that holds it (two 8-bit passes below the
//     values' common high bits). The largest such bound over r is taken, and
//     every CTA gathers its candidate-buffer keys at or above it into a
//     global list. (A key a CTA dropped had top_k larger keys in that CTA's
//     buffer, so at least top_k keys are gathered.)
//  C. If more than f_cap keys passed, digit histograms over all CTAs narrow
//     the bin that holds the top_k-th key (a distributed radix select, a
//     group barrier per round) until the keys at or above the bin fit, and
//     the gather is repeated. Then each CTA ranks a slice of the candidates
//     against all of them (keys are unique, so a key's rank is the number of
//     larger keys) and writes those of rank < top_k to their output slots.

struct FusedSmem {
    unsigned long long qbound[kMaxQG];  // per query: the certified bound of step B
    unsigned long long qmax[kMaxQG];    // and its largest key
    int qn[kMaxQG], qoff[kMaxQG], qtot[kMaxQG];  // gather count / offset, candidates gathered
    unsigned long long lo, hi;  // histogram rounds
    int n, off, above, total, fail;
    int hist[256];
    int wtot[32];  // warp totals of the block scans
};
constexpr uint32_t kFusedHdr = (static_cast<uint32_t>(sizeof(FusedSmem)) + 127u) & ~127u;
// Early steps (one query per group): the streaming epilogue groups (group 0,
// or groups 0-1 taking tiles in turn) hand their row maxima over after about
// f_pub tiles and go on streaming, while the other groups run steps A-B.
// Their scratch: header, the 128 sorted row maxima, the streaming groups' row
// maxima, one query's histograms.
constexpr uint32_t kEarlyBytes = kFusedHdr + 128 * 8 + 2 * 128 * 8 + 2 * kFusedLevels * 256 * 4;
constexpr int kEarlyBar = 6;     // streaming groups arrive, the others wait (all 512 threads)
constexpr int kEarlyGrpBar = 7;  // the early groups among themselves


__device__ __forceinline__ unsigned ld_acquire_u32(const unsigned *ptr) {
    unsigned v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(ptr) : "memory");
    return v;
}

// Barrier of the CTAs of query group g, called by the nthreads threads of a
// CTA that take part (named barrier `bar`; tid 0 among them). Each CTA adds
// one to the group's counter; the n-th barrier of the launch waits for
// n * splits arrivals. The wait is bounded: on timeout it records error code
// 4, sets the abort flag and returns false.
__device__ __noinline__ bool group_sync(const ScoreParams &p, int g, int &nsync, int tid, volatile int *abort_flag,
                           int bar = kEpiBar, int nthreads = kEpiThreads) {
    ++nsync;
    named_bar(bar, nthreads);
    if (tid == 0) {
        unsigned *ctr = p.f_bar + g;
        const unsigned target = static_cast<unsigned>(nsync) * static_cast<unsigned>(p.splits) +
                                (p.fault == 3 && nsync == 1 ? 1u : 0u);
        // release: the CTA's earlier writes (ordered before this thread by the
        // barrier above) are visible to whoever acquires the count
        asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(ctr), "r"(1u) : "memory");
        if (ld_acquire_u32(ctr) < target) {
            const long long t0 = clock64();
            while (ld_acquire_u32(ctr) < target) {
                if (clock64() - t0 > p.wait_limit) {
                    *abort_flag = 1;
                    atomicCAS(&g_dev_error, 0, 4);
                    break;
                }
            }
        }
    }
    named_bar(bar, nthreads);
    return *abort_flag == 0;
}

// A row with no key gets a small stand-in (1..128, below every real key, which
// is >= 2^32) so that all 128 values of a CTA are distinct.
__device__ __forceinline__ unsigned long long row_value(unsigned long long rowmax, int row) {
    return rowmax != 0ull ? rowmax : static_cast<unsigned long long>(128 - row);
}

// Number of entries of a descending list l[0, 32) of distinct values that are > v.
__device__ __forceinline__ int count_above32(const unsigned long long *l, unsigned long long v) {
    int pos = 0;
#pragma unroll
    for (int step = 16; step > 0; step >>= 1)
        if (l[pos + step - 1] > v) pos += step;
    return pos + (l[pos] > v ? 1 : 0);  // pos <= 31 here
}

// Adds this CTA's keys b[0, n) that are >= B to query t's global candidate
// list, counted in slot `attempt`; keys past f_cap are counted, not stored.
// Positions inside the CTA come from a block scan (no shared atomics).
__device__ __forceinline__ void fused_gather(const uint64_t *b, int n, uint64_t B, long long t, int attempt,
                                             FusedSmem *fs, const ScoreParams &p, int tid) {
    constexpr int T = kEpiThreads;
    int mine = 0;
    for (int j = tid; j < n; j += T) mine += b[j] >= B ? 1 : 0;
    int total = 0;
    const int pos0 = block_excl_scan<T>(mine, tid, kEpiBar, fs->wtot, &total);
    if (tid == 0) fs->off = total ? atomicAdd(&p.f_count[t * kFusedAttempts + attempt], total) : 0;
    named_bar(kEpiBar, T);
    int pos = fs->off + pos0;
    uint64_t *dst = p.f_cand + t * p.f_cap;
    for (int j = tid; j < n; j += T) {
        const uint64_t key = b[j];
        if (key >= B) {
            if (pos < p.f_cap) dst[pos] = key;
            ++pos;
        }
    }
}

// Split 0 of a group clears its queries' candidate counters and round
// histograms (read only after the first group barrier).
template <int T>
__device__ __forceinline__ void fused_zero_counts(const ScoreParams &p, long long t_base, int nq, int tid) {
    for (int i = tid; i < nq * kFusedAttempts; i += T) p.f_count[t_base * kFusedAttempts + i] = 0;
    for (int i = tid; i < kFusedRounds * nq * 256; i += T) {
        const int r = i / (nq * 256), rest = i - r * nq * 256;
        p.f_hist[(static_cast<long long>(r) * p.n_q + t_base) * 256 + rest] = 0;
    }
}

// Step A's ranks: srt holds, per query, its four quarters of row maxima,
// each sorted descending ([query][quarter][32]); the value of rank 2^l - 1
// among the 128 becomes the CTA's certificate of level l. T threads, tid < T.
template <int T>
__device__ __forceinline__ void fused_publish(const unsigned long long *srt, int nq, long long t_base, int split,
                                              const ScoreParams &p, int tid) {
    const int S = p.splits;
    for (int e0 = 0; e0 < nq * 128; e0 += T) {
        const int e = e0 + tid;
        if (e < nq * 128) {
            const unsigned long long *q = srt + (e & ~127);
            const int quarter = (e >> 5) & 3;
            const unsigned long long v = srt[e];
            int rank = e & 31;
#pragma unroll
            for (int o = 1; o < 4; ++o) rank += count_above32(q + ((quarter + o) & 3) * 32, v);
            if ((rank & (rank + 1)) == 0)
                // level-major ([row][level][split]): a level's certificates are one contiguous run
                p.f_stats[((t_base + (e >> 7)) * kFusedLevels + (31 - __clz(rank + 1))) * S + split] =
                    v > 255ull ? v : 0ull;
        }
    }
}

// Step B's bounds: fs->qbound / fs->qmax of the group's nq queries from the
// published certificates. For each (query, level l) with c = ceil(top_k /
// 2^l) <= splits, one warp bins the S certificates' scores (as ord values,
// monotone in the score) over [smallest, largest] into 256 bins by a
// monotone map (a larger value never lands in a lower bin); if the bin
// holding the c-th largest has smallest ord m, at least c certificates are
// >= m, so (m << 32) is a lower bound on the query's top_k-th key. The largest
// bound over the levels is taken. T threads on named barrier `bar`; each
// working warp uses 2 KB of lh (lh_bytes in all).
constexpr int kBoundVPL = 5;  // certificates of one level a lane holds: splits <= 160
template <int T>
__device__ __forceinline__ void fused_bound(const ScoreParams &p, FusedSmem *fs, int *lh, int lh_bytes,
                                            long long t_base, int nq, int tid, int bar) {
    constexpr int NW = T / 32;
    const int S = p.splits, K = p.top_k;
    const int lane = tid & 31, warp = tid >> 5;
    const int nwb = min(NW, lh_bytes / 2048);  // warps with scratch
    for (int qi = tid; qi < nq; qi += T) fs->qbound[qi] = 0ull;
    named_bar(bar, T);
    if (warp < nwb) {
        int *hist = lh + warp * 512;  // [256] counts, then [256] smallest ord per bin
        unsigned *minb = reinterpret_cast<unsigned *>(hist + 256);
        for (int pr = warp; pr < nq * kFusedLevels; pr += nwb) {
            const int qi = pr >> 3, l = pr & 7;
            const int c = (K + (1 << l) - 1) >> l;
            if (c > S && l != 0) continue;  // warp-uniform
            const unsigned long long *st = reinterpret_cast<const unsigned long long *>(
                p.f_stats + ((t_base + qi) * kFusedLevels + l) * S);
            uint32_t o[kBoundVPL];
#pragma unroll
            for (int k = 0; k < kBoundVPL; ++k) {
                const int j = lane + 32 * k;
                o[k] = j < S ? static_cast<uint32_t>(__ldcg(st + j) >> 32) : 0u;
            }
            uint32_t lo = ~0u, hi = 0u;
#pragma unroll
            for (int k = 0; k < kBoundVPL; ++k) {
                if (o[k] != 0u) lo = o[k] < lo ? o[k] : lo;
                hi = o[k] > hi ? o[k] : hi;
            }
            lo = __reduce_min_sync(0xFFFFFFFFu, lo);
            hi = __reduce_max_sync(0xFFFFFFFFu, hi);
            if (l == 0 && lane == 0)  // >= the query's largest key
                fs->qmax[qi] = (static_cast<uint64_t>(hi) << 32) | 0xFFFFFFFFull;
            if (c > S || lo > hi) continue;  // no certificate at this level (uniform)
            for (int b = lane; b < 256; b += 32) {
                hist[b] = 0;
                minb[b] = ~0u;
            }
            __syncwarp();
            const float scale = 256.f / (static_cast<float>(hi - lo) + 1.f);
            int nz = 0;
#pragma unroll
            for (int k = 0; k < kBoundVPL; ++k)
                if (o[k] != 0u) {
                    const int bin = min(255, static_cast<int>(static_cast<float>(o[k] - lo) * scale));
                    atomicAdd(&hist[bin], 1);
                    atomicMin(&minb[bin], o[k]);
                    ++nz;
                }
            nz = __reduce_add_sync(0xFFFFFFFFu, nz);
            __syncwarp();
            if (nz >= c) {
                int d, ab, inb;
                scan_digit<8>(hist, c, lane, d, ab, inb);
                uint32_t bound = d >= 0 ? minb[d] : 0u;
                if (d >= 0 && inb > 1) {
                    // a wide bin (the certificates span a wide range, e.g. some of
                    // them -inf): bin its values again over their own range, so the
                    // bound lands next to the c-th largest certificate
                    uint32_t lo2 = ~0u, hi2 = 0u;
#pragma unroll
                    for (int k = 0; k < kBoundVPL; ++k)
                        if (o[k] != 0u &&
                            min(255, static_cast<int>(static_cast<float>(o[k] - lo) * scale)) == d) {
                            lo2 = o[k] < lo2 ? o[k] : lo2;
                            hi2 = o[k] > hi2 ? o[k] : hi2;
                        }
                    lo2 = __reduce_min_sync(0xFFFFFFFFu, lo2);
                    hi2 = __reduce_max_sync(0xFFFFFFFFu, hi2);
                    __syncwarp();
                    for (int bb = lane; bb < 256; bb += 32) {
                        hist[bb] = 0;
                        minb[bb] = ~0u;
                    }
                    __syncwarp();
                    const float scale2 = 256.f / (static_cast<float>(hi2 - lo2) + 1.f);
#pragma unroll
                    for (int k = 0; k < kBoundVPL; ++k)
                        if (o[k] != 0u &&
                            min(255, static_cast<int>(static_cast<float>(o[k] - lo) * scale)) == d) {
                            const int bin = min(255, static_cast<int>(static_cast<float>(o[k] - lo2) * scale2));
                            atomicAdd(&hist[bin], 1);
                            atomicMin(&minb[bin], o[k]);
                        }
                    __syncwarp();
                    int d2, ab2, inb2;
                    scan_digit<8>(hist, c - ab, lane, d2, ab2, inb2);
                    if (d2 >= 0) bound = minb[d2];
                }
                if (lane == 0 && d >= 0)
                    atomicMax(&fs->qbound[qi], static_cast<unsigned long long>(bound) << 32);
            }
            __syncwarp();  // the next pair zeroes the scratch
        }
    }
    named_bar(bar, T);
}

// Steps A-C for the CTA (group g, split) once all its tiles are consumed;
// buf / cnt are its candidate buffers, fs its fused-path header, data a
// shared area of `room` keys (the idle K stages). With REGU the sorted row
// maxima of each query are already in data ([query][quarter][32]);
// otherwise step A builds them from the candidate buffers. With early_done,
// steps A and B already ran (on idle warps, during streaming) and the
// launch has passed its first group barrier.
template <bool REGU>
__device__ __noinline__ void fused_tail(const uint64_t *buf, const int *cnt, FusedSmem *fs, uint64_t *data, int room,
                                           const ScoreParams &p, int g, int split, int tid, volatile int *abort_flag,
                                           bool early_done) {
    constexpr int T = kEpiThreads;
    constexpr int NW = T / 32;
    const int S = p.splits, K = p.top_k, cap = p.cap;
    const long long t_base = static_cast<long long>(g) * p.QG;
    const int nq = static_cast<int>(min(static_cast<long long>(p.QG), p.n_q - t_base));
    unsigned long long *udata = reinterpret_cast<unsigned long long *>(data);
    const int lane = tid & 31, warp = tid >> 5;
    int nsync = early_done ? 1 : 0;

    if (!early_done) {
        // ---- A. certificates
        if (!REGU) {
            for (int i = tid; i < nq * 128; i += T) data[i] = 0ull;
            named_bar(kEpiBar, T);
            for (int qi = 0; qi < nq; ++qi) {
                const uint64_t *b = buf + qi * cap;
                const int n = cnt[qi];
                for (int j = tid; j < n; j += T) {
                    const uint64_t key = b[j];
                    atomicMax(udata + qi * 128 + ((~static_cast<uint32_t>(key)) & 127u),
                              static_cast<unsigned long long>(key));
                }
            }
            named_bar(kEpiBar, T);
            for (int task = warp; task < nq * 4; task += NW) {  // (query, quarter) per warp
                const int row = (task & 3) * 32 + lane;
                unsigned long long *q = udata + (task >> 2) * 128;
                q[row] = warp_sort_desc_u64(row_value(q[row], row), lane);
            }
        }
        named_bar(kEpiBar, T);
        if (split == 0) fused_zero_counts<T>(p, t_base, nq, tid);
        fused_publish<T>(udata, nq, t_base, split, p, tid);
        if (!group_sync(p, g, nsync, tid, abort_flag)) return;
        // ---- B. the bound of each query
        fused_bound<T>(p, fs, reinterpret_cast<int *>(data), room * 8, t_base, nq, tid, kEpiBar);
    }

    // this CTA's keys at or above each query's bound, into the global lists
    for (int qi = tid; qi < nq; qi += T) {
        if (fs->qbound[qi] == 0ull) fs->qbound[qi] = 1ull;  // no certificate: every key is a candidate
        fs->qn[qi] = 0;
    }
    if (tid == 0) fs->n = 0;
    named_bar(kEpiBar, T);
    if (early_done && p.f_reg != nullptr && fs->qbound[0] > 1ull) {
        // One query (early steps ran): each split writes its keys >= B into its own
        // region with plain stores (count first, then the keys, zero-padded), the
        // group meets once, and every CTA loads all regions and ranks its own keys.
        // A region that overflows sends every CTA to the general gather below.
        const int R = p.f_regcap;
        const uint64_t B = fs->qbound[0];
        const int n = cnt[0];
        uint64_t *reg = p.f_reg + (t_base * S + split) * static_cast<long long>(R + 1);
        {
            int c = 0;
            for (int j = tid; j < n; j += T) c += buf[j] >= B ? 1 : 0;
            int mine = 0;
            int pos = block_excl_scan<T>(c, tid, kEpiBar, fs->wtot, &mine);
            for (int j = tid; j < n; j += T) {
                const uint64_t key = buf[j];
                if (key >= B) {
                    if (pos < R) reg[1 + pos] = key;
                    ++pos;
                }
            }
            for (int j = mine + tid; j < R; j += T) reg[1 + j] = 0ull;
            if (tid == 0) reg[0] = static_cast<uint64_t>(mine);
            if (tid == 0) fs->n = mine;
        }
        if (!group_sync(p, g, nsync, tid, abort_flag)) return;
        const int mine = fs->n;
        // every region of the query (headers are counts, far below any real key,
        // which is >= 2^32; empty slots are 0)
        const int W = S * (R + 1);
        const unsigned long long *src =
            reinterpret_cast<const unsigned long long *>(p.f_reg + t_base * S * static_cast<long long>(R + 1));
        constexpr int kLd = 8;  // loads in flight per thread
        bool ovf = false;
        int c = 0;  // this thread's candidates
        for (int j0 = 0; j0 < W; j0 += kLd * T) {
            unsigned long long r[kLd];
#pragma unroll
            for (int u = 0; u < kLd; ++u) {
                const int j = j0 + u * T + tid;
                r[u] = j < W ? __ldcg(src + j) : 0ull;
            }
#pragma unroll
            for (int u = 0; u < kLd; ++u) {
                const int j = j0 + u * T + tid;
                if (j < W) {
                    udata[j] = r[u];
                    if (r[u] > 0xFFFFFFFFull) ++c;                                  // a key
                    else if (r[u] > static_cast<unsigned long long>(R)) ovf = true;  // a header past R
                }
            }
        }
        if (!named_bar_or(kEpiBar, T, ovf)) {
            // the candidates, packed after the regions (positions from a block scan)
            unsigned long long *cand = udata + W;
            int total = 0;
            int pos = block_excl_scan<T>(c, tid, kEpiBar, fs->wtot, &total);
            for (int j0 = 0; j0 < W; j0 += kLd * T)
#pragma unroll
                for (int u = 0; u < kLd; ++u) {
                    const int j = j0 + u * T + tid;
                    if (j < W && udata[j] > 0xFFFFFFFFull) cand[pos++] = udata[j];
                }
            named_bar(kEpiBar, T);
            const unsigned long long *own = udata + split * (R + 1) + 1;
            const long long t = t_base;
            for (int ci = warp; ci < mine; ci += NW) {
                const unsigned long long x = own[ci];
                int r = 0, r1 = 0, r2 = 0, r3 = 0;  // four independent chains
                int y = lane;
                for (; y + 96 < total; y += 128) {
                    r += cand[y] > x ? 1 : 0;
                    r1 += cand[y + 32] > x ? 1 : 0;
                    r2 += cand[y + 64] > x ? 1 : 0;
                    r3 += cand[y + 96] > x ? 1 : 0;
                }
                for (; y < total; y += 32) r += cand[y] > x ? 1 : 0;
                r = __reduce_add_sync(0xFFFFFFFFu, r + r1 + r2 + r3);
                if (lane == 0 && r < K) {
                    int32_t idx;
                    float sc;
                    decode_key(x, idx, sc);
                    p.out_idx[t * K + r] = idx;
                    p.out_score[t * K + r] = sc;
                }
            }
            if (split == 0)  // (a certified bound admits at least top_k keys: no padding is due)
                for (int j = total + tid; j < K; j += T) {
                    p.out_idx[t * K + j] = -1;
                    p.out_score[t * K + j] = __uint_as_float(0xFF800000u);
                }
            return;
        }
        // a region overflowed (uniform): the general path below, from a clean count
        if (tid == 0) fs->n = 0;
        named_bar(kEpiBar, T);
    }
    {
        // each query's keys >= its bound: positions within the CTA from a scan per query,
        // then one round of global offset atomics for all the queries together
        int mybase[kMaxQG];
        for (int qi = 0; qi < nq; ++qi) {
            const uint64_t *b = buf + qi * cap;
            const uint64_t B = fs->qbound[qi];
            int c = 0;
            for (int j = tid; j < cnt[qi]; j += T) c += b[j] >= B ? 1 : 0;
            int tot = 0;
            mybase[qi] = block_excl_scan<T>(c, tid, kEpiBar, fs->wtot, &tot);
            if (tid == 0) fs->qn[qi] = tot;
        }
        named_bar(kEpiBar, T);
        for (int qi = tid; qi < nq; qi += T)
            fs->qoff[qi] = fs->qn[qi] ? atomicAdd(&p.f_count[(t_base + qi) * kFusedAttempts], fs->qn[qi]) : 0;
        named_bar(kEpiBar, T);
        for (int qi = 0; qi < nq; ++qi) {
            const uint64_t *b = buf + qi * cap;
            const uint64_t B = fs->qbound[qi];
            uint64_t *dst = p.f_cand + (t_base + qi) * p.f_cap;
            int pos = fs->qoff[qi] + mybase[qi];
            for (int j = tid; j < cnt[qi]; j += T) {
                const uint64_t key = b[j];
                if (key >= B) {
                    if (pos < p.f_cap) dst[pos] = key;
                    ++pos;
                }
            }
        }
    }
    if (!group_sync(p, g, nsync, tid, abort_flag)) return;

    // ---- C. narrow oversized candidate sets, then rank and write
    for (int qi = tid; qi < nq; qi += T) fs->qtot[qi] = __ldcg(&p.f_count[(t_base + qi) * kFusedAttempts]);
    named_bar(kEpiBar, T);
    for (int qi = 0; qi < nq; ++qi) {
        if (fs->qtot[qi] <= p.f_cap) continue;  // uniform: every CTA read the same totals
        const long long t = t_base + qi;
        uint64_t lo = fs->qbound[qi], hi = fs->qmax[qi];
        int above = 0;  // keys > hi
        int attempt = 0;
        const uint64_t *b = buf + qi * cap;
        const int n = cnt[qi];
        for (int r = 0; r < kFusedRounds && attempt == 0; ++r) {
            const uint64_t diff = lo ^ hi;
            const int hb = diff ? 63 - __clzll(static_cast<long long>(diff)) : 0;
            const int shift = hb >= 7 ? hb - 7 : 0;
            for (int i = tid; i < 256; i += T) fs->hist[i] = 0;
            named_bar(kEpiBar, T);
            for (int j = tid; j < n; j += T) {
                const uint64_t key = b[j];
                if (key >= lo && key <= hi) atomicAdd(&fs->hist[(key >> shift) & 255u], 1);
            }
            named_bar(kEpiBar, T);
            int *gh = p.f_hist + (static_cast<long long>(r) * p.n_q + t) * 256;
            for (int i = tid; i < 256; i += T)
                if (fs->hist[i]) atomicAdd(gh + i, fs->hist[i]);
            if (!group_sync(p, g, nsync, tid, abort_flag)) return;
            for (int i = tid; i < 256; i += T) fs->hist[i] = __ldcg(gh + i);
            named_bar(kEpiBar, T);
            if (warp == 0) {
                int d, ab, inb;
                scan_digit<8>(fs->hist, K - above, lane, d, ab, inb);
                if (lane == 0) {
                    if (d < 0) {
                        fs->fail = 1;
                    } else {
                        const uint64_t span = shift + 8 >= 64 ? ~0ull : ((1ull << (shift + 8)) - 1ull);
                        const uint64_t base = (lo & ~span) | (static_cast<uint64_t>(d) << shift);
                        const uint64_t top = base | ((1ull << shift) - 1ull);
                        fs->fail = 0;
                        fs->lo = base > lo ? base : lo;
                        fs->hi = top < hi ? top : hi;
                        fs->above = above + ab;
                        fs->total = above + ab + inb;
                    }
                }
            }
            named_bar(kEpiBar, T);
            if (fs->fail) break;
            lo = fs->lo;
            hi = fs->hi;
            above = fs->above;
            if (fs->total <= p.f_cap) attempt = r + 1;
            named_bar(kEpiBar, T);
        }
        if (attempt == 0) {  // cannot happen for unique keys: after 8 rounds the bin is one key
            if (tid == 0) atomicCAS(&g_dev_error, 0, 5);
            return;
        }
        fused_gather(b, n, lo, t, attempt, fs, p, tid);
        if (!group_sync(p, g, nsync, tid, abort_flag)) return;
        if (tid == 0) {
            int tot = __ldcg(&p.f_count[t * kFusedAttempts + attempt]);
            if (tot > p.f_cap) {  // cannot happen: the histograms count exactly the keys gathered
                atomicCAS(&g_dev_error, 0, 5);
                tot = p.f_cap;
            }
            fs->qtot[qi] = tot;
        }
        named_bar(kEpiBar, T);
    }
    // ranking, as many queries at a time as the data area holds
    for (int q0 = 0; q0 < nq;) {
        int q1 = q0, used = 0;
        while (q1 < nq && used + fs->qtot[q1] <= room) used += fs->qtot[q1++];
        // every CTA loads the chunk's candidates, eight loads in flight per thread
        // (query qi's occupy data[start, start + qtot[qi]) with the chunk's queries packed)
        for (int j0 = 0; j0 < used; j0 += 8 * T) {
            unsigned long long r[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const int j = j0 + u * T + tid;
                r[u] = 0ull;
                if (j < used) {
                    int qi = q0, start = 0;
                    while (j >= start + fs->qtot[qi]) start += fs->qtot[qi++];
                    r[u] = __ldcg(reinterpret_cast<const unsigned long long *>(p.f_cand + (t_base + qi) * p.f_cap) +
                                  (j - start));
                }
            }
#pragma unroll
            for (int u = 0; u < 8; ++u)
                if (j0 + u * T + tid < used) data[j0 + u * T + tid] = r[u];
        }
        named_bar(kEpiBar, T);
        int base;
        base = 0;
        for (int qi = q0; qi < q1; ++qi) {
            const int n = fs->qtot[qi];
            const uint64_t *cs = data + base;
            const long long t = t_base + qi;
            const int per = (n + S - 1) / S;
            const int lo = split * per, hi = min(n, lo + per);
            for (int c = lo + warp; c < hi; c += NW) {
                const uint64_t x = cs[c];
                int r = 0, r1 = 0, r2 = 0, r3 = 0;  // four independent chains
                int y = lane;
                for (; y + 96 < n; y += 128) {
                    r += cs[y] > x ? 1 : 0;
                    r1 += cs[y + 32] > x ? 1 : 0;
                    r2 += cs[y + 64] > x ? 1 : 0;
                    r3 += cs[y + 96] > x ? 1 : 0;
                }
                for (; y < n; y += 32) r += cs[y] > x ? 1 : 0;
                r = __reduce_add_sync(0xFFFFFFFFu, r + r1 + r2 + r3);
                if (lane == 0 && r < K) {
                    int32_t idx;
                    float sc;
                    decode_key(x, idx, sc);
                    p.out_idx[t * K + r] = idx;
                    p.out_score[t * K + r] = sc;
                }
            }
            if (split == 0)
                for (int j = n + tid; j < K; j += T) {
                    p.out_idx[t * K + j] = -1;
                    p.out_score[t * K + j] = __uint_as_float(0xFF800000u);
                }
            base += n;
        }
        named_bar(kEpiBar, T);
        q0 = q1;
    }
}

// Steps A-B on the early groups: T of their threads, etid < T. nstream
// streaming groups left their row maxima in comb[g][128].
template <int T>
__device__ __noinline__ void early_steps(const ScoreParams &p, uint8_t *early, int nstream, int g, int split,
                                            int etid, volatile int *abort_flag, volatile unsigned long long *live) {
    FusedSmem *efs = reinterpret_cast<FusedSmem *>(early);
    unsigned long long *es = reinterpret_cast<unsigned long long *>(early + kFusedHdr);
    const unsigned long long *comb = es + 128;
    int *elh = reinterpret_cast<int *>(early + kFusedHdr + 3 * 128 * 8);
    const int lane = etid & 31, w = etid >> 5;
    if (w < 4) {  // quarter w: the rows' maxima over the streaming groups, sorted across the warp
        const int row = w * 32 + lane;
        unsigned long long v = comb[row];
        for (int g2 = 1; g2 < nstream; ++g2) v = comb[g2 * 128 + row] > v ? comb[g2 * 128 + row] : v;
        es[row] = warp_sort_desc_u64(row_value(v, row), lane);
    }
    named_bar(kEarlyGrpBar, T);
    const long long t0 = static_cast<long long>(g) * p.QG;
    if (split == 0) fused_zero_counts<T>(p, t0, 1, etid);
    fused_publish<T>(es, 1, t0, split, p, etid);
    int nsync = 0;
    if (group_sync(p, g, nsync, etid, abort_flag, kEarlyGrpBar, T)) {
        fused_bound<T>(p, efs, elh, 2 * kFusedLevels * 256 * 4, t0, 1, etid, kEarlyGrpBar);
        // the streaming groups keep only keys at or above it from here on
        if (etid == 0) *live = efs->qbound[0];
    }
}

template <int H, bool FUSED>
__global__ void __maxnreg__(96)
    score_select_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_q,
                        const __grid_constant__ ScoreParams p) {
    extern __shared__ uint8_t smem_raw[];
    // 1024-byte aligned base, by pointer arithmetic on the shared array so that
    // the compiler keeps every derived pointer in the shared address space
    uint8_t *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    const SmemLayout L = smem_layout(p.D, p.N, p.QG, H, p.kstages, p.cap, p.f_early ? kEarlyBytes : 0u);
    uint8_t *early = smem + L.early_off;  // (f_early) FusedSmem, sorted row maxima, histograms
    uint8_t *k_smem = smem + L.k_off;
    uint8_t *q_smem = smem + L.q_off;
    float *w_s = reinterpret_cast<float *>(smem + L.w_off);
    uint64_t *buf = reinterpret_cast<uint64_t *>(smem + L.buf_off);
    Misc *m = reinterpret_cast<Misc *>(smem + L.misc_off);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int g = blockIdx.x % p.n_groups;
    const int split = blockIdx.x / p.n_groups;
    constexpr int ne_threads = kEpiThreads;
    const long long t_base = static_cast<long long>(g) * p.QG;
    const bool ranged = p.row_lo != nullptr;

    // Nothing before the dependency wait below touches global memory: under a
    // programmatic launch this prologue overlaps the previous grid's tail, and
    // the inputs (and the workspace) are read only once that grid is done.
    const int nchunk = p.D * p.esize / 128;  // operands arrive in 128-byte column chunks
    const int cw = 128 / p.esize;            // (64 16-bit or 128 8-bit elements)
    const uint32_t tile_bytes = static_cast<uint32_t>(kBM * p.D * p.esize);
    if (threadIdx.x == 0) {
        for (int s = 0; s < p.kstages; ++s) {
            mbar_init(&m->k_full[s], 1);
            mbar_init(&m->k_empty[s], 1);
        }
        for (int a = 0; a < p.acc_stages; ++a) {
            mbar_init(&m->acc_full[a], 1);
            mbar_init(&m->acc_empty[a], 4 * active_groups(p.QG));
        }
        mbar_init(&m->q_full, 1);
        mbar_init(&m->mma_done, 1);
        mbar_init(&m->never, 1);
        m->abort_flag = 0;
        m->live_bound = 0ull;
        fence_mbar_init();
        tma_prefetch_desc(&tm_k);
        tma_prefetch_desc(&tm_q);
        asm volatile("griddepcontrol.wait;" ::: "memory");
        // this CTA's tiles: its split of the keys, or, with visible ranges that
        // each hold at least top_k keys, its split of the tiles the group's
        // ranges touch (keys outside every range score -inf and cannot reach
        // the output)
        int gt0 = 0, gt1 = p.n_tiles, tps = p.tiles_per_split;
        if (ranged) {
            long long ulo = p.n_kv, uhi = 0;
            bool narrow = true;
            for (int qi = 0; qi < p.QG; ++qi) {
                const long long t = t_base + qi;
                long long lo = 0, hi = 0;
                if (t < p.n_q) {
                    lo = p.row_lo[t];
                    hi = p.row_hi[t];
                    lo = lo < 0 ? 0 : (lo > p.n_kv ? p.n_kv : lo);
                    hi = hi < lo ? lo : (hi > p.n_kv ? p.n_kv : hi);
                    if (hi - lo < p.top_k) narrow = false;  // its lowest-index masked keys are needed too
                    ulo = lo < ulo ? lo : ulo;
                    uhi = hi > uhi ? hi : uhi;
                }
                m->qlo[qi] = static_cast<int>(lo);
                m->qhi[qi] = static_cast<int>(hi);
            }
            if (narrow && uhi > ulo) {
                gt0 = static_cast<int>(ulo / kBM);
                gt1 = static_cast<int>((uhi + kBM - 1) / kBM);
                tps = (gt1 - gt0 + p.splits - 1) / p.splits;
            }
        } else {
            for (int qi = 0; qi < p.QG; ++qi) {  // every key inside (the dense mask decides)
                m->qlo[qi] = 0;
                m->qhi[qi] = 0x7FFFFFFF;
            }
        }
        const int a = gt0 + split * tps;
        m->tile0 = a;
        m->ntl = max(0, min(a + tps, gt1) - a);
        // the first loads leave before the block barrier: q, then up to kstages K tiles
        const int ntl0 = m->ntl;
        if (ntl0 > 0) {
            mbar_arrive_expect_tx(&m->q_full, static_cast<uint32_t>(p.N * p.D * p.esize));
            for (int c = 0; c < nchunk; ++c)
                tma_load_2d(q_smem + c * p.N * 128, &tm_q, c * cw, static_cast<int>(t_base * H), &m->q_full);
        }
        for (int i = 0; i < ntl0 && i < p.kstages; ++i) {
            mbar_arrive_expect_tx(&m->k_full[i], tile_bytes);
            for (int c = 0; c < nchunk; ++c)
                tma_load_2d(k_smem + i * L.stage_bytes + c * kBM * 128, &tm_k, c * cw, (m->tile0 + i) * kBM,
                            &m->k_full[i]);
        }
    }
    if (warp == 1) {
        tmem_alloc(&m->tmem_base, p.tmem_cols);
        tmem_relinquish();
    }
    if (warp >= 2) {
        const int etid = threadIdx.x - 64;
        for (int i = etid; i < p.QG; i += ne_threads) m->cnt[i] = 0;
        asm volatile("griddepcontrol.wait;" ::: "memory");
        for (int i = etid; i < p.QG * H; i += ne_threads) {
            const long long t = t_base + i / H;
            // with 8-bit operands w[t,h] relu(q_scale[t,h] x) = (w[t,h] q_scale[t,h]) relu(x)
            // (scales are non-negative), so the q scale rides on the head weight
            const float qsc = (t < p.n_q && p.q_scale != nullptr) ? p.q_scale[t * H + (i % H)] : 1.f;
            w_s[i] = (t < p.n_q) ? p.w[t * H + (i % H)] * qsc : 0.f;
        }
    }
    asm volatile("griddepcontrol.wait;" ::: "memory");  // (every thread: it reads global memory later)
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = m->tmem_base;
    const int tile0 = m->tile0;
    const int ntl = m->ntl;
    volatile int *abort_flag = &m->abort_flag;

    if (warp == 0) {
        // ------------------------------------------------------ TMA producer
        if (lane == 0) {
            // q and the first kstages tiles are already on their way (prologue)
            int issued = ntl < p.kstages ? ntl : p.kstages;
            int s = issued % p.kstages;
            uint32_t ph = static_cast<uint32_t>(issued / p.kstages) & 1u;
            for (int i = issued; i < ntl; ++i) {
                if (i >= p.kstages && !mbar_wait(&m->k_empty[s], ph ^ 1u, abort_flag, 1, p.wait_limit)) break;
                mbar_arrive_expect_tx(&m->k_full[s], tile_bytes);
                uint8_t *dst = k_smem + s * L.stage_bytes;
                for (int c = 0; c < nchunk; ++c)
                    tma_load_2d(dst + c * kBM * 128, &tm_k, c * cw, (tile0 + i) * kBM, &m->k_full[s]);
                issued = i + 1;
                if (++s == p.kstages) {
                    s = 0;
                    ph ^= 1u;
                }
            }
            // wait (bounded) for loads still in flight before the CTA may exit
            const int first = max(0, issued - p.kstages);
            for (int i = first; i < issued; ++i) {
                const int s = i % p.kstages;
                const uint32_t ph = static_cast<uint32_t>(i / p.kstages) & 1u;
                int dummy = 0;
                mbar_wait(&m->k_full[s], ph, &dummy, 1, p.wait_limit);
            }
            if (ntl > 0) {
                int dummy = 0;
                mbar_wait(&m->q_full, 0, &dummy, 1, p.wait_limit);
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        // ------------------------------------------------------- MMA issuer
        if (lane == 0) {
            // descriptors of the stage bases; an MMA's operands are at fixed offsets from them
            // (the address field is the low 14 bits of addr >> 4: adding offset >> 4 moves it)
            const uint64_t q_desc = smem_desc_sw128(smem_u32(q_smem));
            const uint64_t k_desc = smem_desc_sw128(smem_u32(k_smem));
            // one MMA per 32 bytes of a row (K = 16 for 16-bit operands, 32 for E4M3), four per
            // 128-byte column chunk: D * esize / 128 chunks (1 or 2); the second chunk's
            // operands are a chunk of rows further on
            const bool f8 = p.esize == 1;
            const bool two_chunks = p.D * p.esize == 256;
            const uint64_t b_step_k = static_cast<uint64_t>(kBM * 128) >> 4;
            const uint64_t b_step_q = static_cast<uint64_t>(p.N * 128) >> 4;
            bool ok = ntl == 0 || mbar_wait(&m->q_full, 0, abort_flag, 2, p.wait_limit);
            tc_fence_after();
            int s = 0, a = 0;
            uint32_t kph = 0u, aph = 0u;
            for (int i = 0; ok && i < ntl; ++i) {
                if (!mbar_wait(&m->k_full[s], kph, abort_flag, 2, p.wait_limit)) break;
                if (i >= p.acc_stages && !mbar_wait(&m->acc_empty[a], aph ^ 1u, abort_flag, 2, p.wait_limit))
                    break;
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(a * p.N);
                const uint64_t ks = k_desc + ((s * L.stage_bytes) >> 4);
                if (f8) {
                    umma_quad<true>(d_tmem, ks, q_desc, p.idesc, 0u);  // D = 128 codes: one chunk
                } else {
                    umma_quad<false>(d_tmem, ks, q_desc, p.idesc, 0u);
                    if (two_chunks) umma_quad<false>(d_tmem, ks + b_step_k, q_desc + b_step_q, p.idesc, 1u);
                }
                umma_commit(&m->k_empty[s]);
                umma_commit(&m->acc_full[a]);
                if (++s == p.kstages) {
                    s = 0;
                    kph ^= 1u;
                }
                if (++a == p.acc_stages) {
                    a = 0;
                    aph ^= 1u;
                }
            }
            // every MMA this thread issued has finished before the CTA may free its
            // tensor memory (on an abort some may still be running here)
            umma_commit(&m->mma_done);
            int dummy = 0;
            mbar_wait(&m->mma_done, 0, &dummy, 2, p.wait_limit);
        }
        __syncwarp();
    } else {
        // ---------------------------------------------------------- epilogue
        const int e = warp - 2;
        const int quarter = warp & 3;
        const int grp = e >> 2;                    // epilogue group
        const int gtid = (e & 3) * 32 + lane;      // thread index within the group
        const int gbar = 2 + grp;                  // the group's named barrier
        const int qpw = queries_per_group(p.QG);
        const int q_lo = grp * qpw;
        const int q_hi = min(p.QG, q_lo + qpw);
        const int row = quarter * 32 + lane;
        const int cap = p.cap;
        constexpr int MAXQPW = H >= 64 ? 1 : 64 / H;   // queries per group at most
        constexpr int CUT_R = kSortMax / 128;          // keys per thread a group cut holds in registers
        CutScratch<kCutDB, 4> *cs = &m->cut[grp];
        // running threshold of each of my queries (keys above it are candidates)
        uint64_t thr[MAXQPW];
#pragma unroll
        for (int qq = 0; qq < MAXQPW; ++qq) thr[qq] = 0ull;
        // one-launch path with at most two queries per group: each thread's row
        // maximum per query, for the certificates
        constexpr bool REGU = FUSED && MAXQPW <= 2;
        unsigned long long umx[REGU ? MAXQPW : 1];
#pragma unroll
        for (int qq = 0; qq < (REGU ? MAXQPW : 1); ++qq) umx[qq] = 0ull;
        bool ok = true;
        // one query and no candidate cut possible (all of a CTA's keys fit its
        // buffer): npar groups take the tiles in turn (group g: tiles g,
        // g + npar, ...) and append to the one buffer. Planned, or found here:
        // with visible ranges a CTA streams only the tiles its range touches,
        // which the plan does not know
        int npar = 0;
        if (p.QG == 1) {
            if (p.tilepar != 0) npar = p.tilepar;
            else if (static_cast<long long>(m->ntl) * kBM + kBM <= cap) npar = p.f_early != 0 ? 2 : 4;
        }
        const int nstream = npar > 0 ? npar : 1;  // epilogue groups that stream
        // early steps: each streaming group hands its row maxima to the other
        // groups once, after about f_pub tiles or when it stops streaming,
        // whichever is first (the others wait on a hardware barrier, so it must arrive)
        constexpr bool EARLY = REGU;
        const bool early_on = EARLY && p.f_early != 0 && p.QG == 1 && nstream < kEPG;
        bool published = false;
        auto early_publish = [&]() {
            unsigned long long *comb = reinterpret_cast<unsigned long long *>(early + kFusedHdr) + 128;
            comb[grp * 128 + row] = umx[0];
            __syncwarp();
            asm volatile("bar.arrive %0, %1;" ::"r"(kEarlyBar), "r"(kEpiThreads) : "memory");
            published = true;
        };

        // sum_h w[t,h] * relu(S[h]) of query qi for my key row, from accumulator
        // column base tacc, in 16-column chunks
        auto head_sum = [&](uint32_t tacc, int qi) {
            const float4 *w4 = reinterpret_cast<const float4 *>(w_s + qi * H);
            uint64_t acc0 = 0ull, acc1 = 0ull, accx = 0ull;
            float acca0 = 0.f, acca1 = 0.f;
            // chunks of CW columns, each loaded and waited for before it is summed
            // (two waits per query for H = 64: the warp stalls on fewer loads)
            constexpr int CW = H < 32 ? H : 32;
            uint32_t xa[CW];
#pragma unroll
            for (int c = 0; c < H; c += CW) {
                uint32_t *cur = xa;
                tmem_ld<CW>(tacc + qi * H + c, xa);
                tmem_wait_ld_dep<CW>(xa);
                // first half of the chunk: w * max(x, 0) (max on the ALU pipe)
#pragma unroll
                for (int h = 0; h < CW / 2; h += 4) {
                    const float4 wv = w4[(c + h) / 4];
                    const uint64_t r01 =
                        pack_f32x2(fmaxf(__uint_as_float(cur[h]), 0.f), fmaxf(__uint_as_float(cur[h + 1]), 0.f));
                    const uint64_t r23 =
                        pack_f32x2(fmaxf(__uint_as_float(cur[h + 2]), 0.f), fmaxf(__uint_as_float(cur[h + 3]), 0.f));
                    acc0 = fma_f32x2(pack_f32x2(wv.x, wv.y), r01, acc0);
                    acc1 = fma_f32x2(pack_f32x2(wv.z, wv.w), r23, acc1);
                }
                // second half: w * max(x, 0) = (w x + w |x|) / 2, all on the FMA pipe
                // (the halving is applied once, exactly, at the end)
#pragma unroll
                for (int h = CW / 2; h < CW; h += 4) {
                    const float4 wv = w4[(c + h) / 4];
                    accx = fma_f32x2(pack_f32x2(wv.x, wv.y), pack_f32x2(__uint_as_float(cur[h]), __uint_as_float(cur[h + 1])),
                                     accx);
                    accx = fma_f32x2(pack_f32x2(wv.z, wv.w),
                                     pack_f32x2(__uint_as_float(cur[h + 2]), __uint_as_float(cur[h + 3])), accx);
                    acca0 = fmaf(wv.x, fabsf(__uint_as_float(cur[h])), acca0);
                    acca1 = fmaf(wv.y, fabsf(__uint_as_float(cur[h + 1])), acca1);
                    acca0 = fmaf(wv.z, fabsf(__uint_as_float(cur[h + 2])), acca0);
                    acca1 = fmaf(wv.w, fabsf(__uint_as_float(cur[h + 3])), acca1);
                }
            }
            return (sum_f32x2(acc0) + sum_f32x2(acc1)) + 0.5f * (sum_f32x2(accx) + (acca0 + acca1));
        };
        const bool tilepar = npar > 0;

        if (tilepar && grp < npar) {
            const uint16_t *mrow0 = (p.mask != nullptr && t_base < p.n_q) ? p.mask + t_base * p.n_kv : nullptr;
            auto mask_bits = [&](int i) -> uint16_t {
                const long long s = static_cast<long long>(tile0 + i) * kBM + row;
                return (mrow0 != nullptr && i < ntl && s < p.n_kv) ? __ldg(mrow0 + s) : static_cast<uint16_t>(0);
            };
            uint16_t mnext = mask_bits(grp);
            for (int i = grp; i < ntl; i += npar) {
                const int a = i % p.acc_stages;
                const uint32_t aph = static_cast<uint32_t>(i / p.acc_stages) & 1u;
                const long long s = static_cast<long long>(tile0 + i) * kBM + row;
                const bool s_ok = s < p.n_kv;
                const uint16_t mbits = mnext;  // loaded one of this group's tiles ago
                mnext = mask_bits(i + npar);
                // key scale (8-bit operands): relu(k_scale[s] x) = k_scale[s] relu(x), so it
                // multiplies the head sum; issued before the wait, used after it
                const float ksc = (p.k_scale != nullptr && s_ok) ? __ldg(p.k_scale + s) : 1.f;
                ok = mbar_wait(p.fault == 2 ? &m->never : &m->acc_full[a], aph, abort_flag, 3, p.wait_limit);
                ok = __all_sync(0xFFFFFFFFu, ok);  // warp-uniform before the .sync.aligned TMEM loads
                tc_fence_after();
                if (!ok) break;
                const bool outside = s < m->qlo[0] || s >= m->qhi[0];  // as in the per-group loop
                const bool hidden = __all_sync(0xFFFFFFFFu, outside || mbits == kF16NegInf);
                const float hs = hidden ? 0.f
                                        : head_sum(tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) +
                                                       static_cast<uint32_t>(a * p.N),
                                                   0);
                const float score =
                    (hidden || outside) ? __uint_as_float(0xFF800000u) : fmaf(hs, ksc, f16_bits_to_float(mbits));
                const bool valid = s_ok && t_base < p.n_q;
                const uint64_t key = valid ? make_key(score, static_cast<uint32_t>(s)) : 0ull;
                if (REGU) umx[0] = key > umx[0] ? key : umx[0];
                // once the early groups hold the certified bound, keys below it cannot
                // reach the output (a lane may still see 0 for a while: it keeps more)
                const bool keep =
                    !early_on || key >= *reinterpret_cast<volatile unsigned long long *>(&m->live_bound);
                warp_append(buf, &m->cnt[0], key, valid && keep, lane);
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&m->acc_empty[a]);
                if (early_on && !published && i + npar >= p.f_pub) early_publish();
            }
            if (early_on && !published) early_publish();
        } else if (!tilepar && q_lo < q_hi) {
            // mask rows of my queries (null: no mask or no such query), advanced one
            // tile per step; values are loaded two tiles before they are used
            const uint16_t *mrow[MAXQPW];
#pragma unroll
            for (int qq = 0; qq < MAXQPW; ++qq) {
                const long long t = t_base + q_lo + qq;
                mrow[qq] = (p.mask != nullptr && q_lo + qq < q_hi && t < p.n_q)
                               ? p.mask + t * p.n_kv + static_cast<long long>(tile0) * kBM + row
                               : nullptr;
            }
            const long long s_first = static_cast<long long>(tile0) * kBM + row;
            // mask bits of tile i (+0.0 where there is none); converted only where
            // used, so that a load is waited for one tile after it was issued
            auto load_mask = [&](int i, uint16_t *mv) {
                const bool in = i < ntl && s_first + static_cast<long long>(i) * kBM < p.n_kv;
#pragma unroll
                for (int qq = 0; qq < MAXQPW; ++qq) mv[qq] = (in && mrow[qq] != nullptr) ? __ldg(mrow[qq] + i * kBM) : 0;
            };
            uint16_t mnext[MAXQPW];
            load_mask(0, mnext);
            int a = 0;            // accumulator stage of tile i
            uint32_t aph = 0u;    // and its phase parity
            if (p.qbound != nullptr) {
                // what the query's other splits have certified so far (the splits of a group run
                // one after another, blockIdx = split * n_groups + group): keys below it cannot
                // reach the output, so they are not appended (a later cut keeps its own bound)
#pragma unroll
                for (int qq = 0; qq < MAXQPW; ++qq) {
                    const long long t = t_base + q_lo + qq;
                    if (q_lo + qq < q_hi && t < p.n_q) {
                        const unsigned long long qb = __ldcg(p.qbound + t);
                        if (qb > thr[qq] + 1ull) thr[qq] = qb - 1ull;
                    }
                }
            }
            for (int i = 0; i < ntl; ++i) {
                const long long s = s_first + static_cast<long long>(i) * kBM;
                const bool s_ok = s < p.n_kv;
                if (early_on) {  // the certified bound, once known, filters appends as a cut would
                    const unsigned long long lb = *reinterpret_cast<volatile unsigned long long *>(&m->live_bound);
                    if (lb > thr[0] + 1ull) thr[0] = lb - 1ull;
                }
                uint16_t mval[MAXQPW];  // loaded one tile ago
#pragma unroll
                for (int qq = 0; qq < MAXQPW; ++qq) mval[qq] = mnext[qq];
                load_mask(i + 1, mnext);
                const float ksc = (p.k_scale != nullptr && s_ok) ? __ldg(p.k_scale + s) : 1.f;  // as above
                ok = mbar_wait(p.fault == 2 ? &m->never : &m->acc_full[a], aph, abort_flag, 3, p.wait_limit);
                ok = __all_sync(0xFFFFFFFFu, ok);  // warp-uniform before the .sync.aligned TMEM loads
                tc_fence_after();
                bool overflow = false;
                if (ok) {
                    const uint32_t tacc = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) +
                                          static_cast<uint32_t>(a * p.N);
#pragma unroll
                    for (int qq = 0; qq < MAXQPW; ++qq) {
                        const int qi = q_lo + qq;
                        if (qi < q_hi) {
                            const long long t = t_base + qi;
                            // a warp whose 32 keys are all masked for this query skips the sum:
                            // the score is -inf whatever it is (inputs are finite)
                            // outside the query's visible range (ranges form; never with a dense mask)
                            const bool outside = s < m->qlo[qi] || s >= m->qhi[qi];
                            const bool hidden = __all_sync(0xFFFFFFFFu, outside || mval[qq] == kF16NegInf);
                            // (the sum's TMEM loads are warp-wide: taken or skipped by the whole warp)
                            const float hs = hidden ? 0.f : head_sum(tacc, qi);
                            const float score = (hidden || outside) ? __uint_as_float(0xFF800000u)
                                                                    : fmaf(hs, ksc, f16_bits_to_float(mval[qq]));
                            const bool valid = s_ok && t < p.n_q;
                            const uint64_t key = valid ? make_key(score, static_cast<uint32_t>(s)) : 0ull;
                            if (REGU) umx[REGU ? qq : 0] = key > umx[REGU ? qq : 0] ? key : umx[REGU ? qq : 0];
                            const int after =
                                warp_append(buf + qi * cap, &m->cnt[qi], key, valid && key > thr[qq], lane);
                            // the last warp to append sees the final count, so this vote is exact
                            overflow |= after > cap - kBM;
                        }
                    }
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&m->acc_empty[a]);
                if (++a == p.acc_stages) {
                    a = 0;
                    aph ^= 1u;
                }
                // one group barrier per tile in the common case: it orders this tile's
                // appends before any cut and tells the group whether a cut (or an abort) is due
                if (named_bar_or(gbar, 128, overflow || !ok || *abort_flag != 0)) {
                    if (named_bar_or(gbar, 128, !ok || *abort_flag != 0)) {
                        ok = false;
                        break;
                    }
#pragma unroll
                    for (int qq = 0; qq < MAXQPW; ++qq) {
                        const int qi = q_lo + qq;
                        if (qi < q_hi) {
                            const int n = m->cnt[qi];  // stable: the group appends nothing until the cut is done
                            if (n > cap - kBM) {
                                uint64_t mk;
                                group_cut<CUT_R, kCutDB, 4>(buf + qi * cap, &m->cnt[qi], n, p.top_k, 64, false, gtid,
                                                            gbar, cs, &mk);
                                // the cut keeps >= top_k keys, all >= mk: a bound for the other splits
                                if (p.qbound != nullptr && gtid == 0 && t_base + qi < p.n_q)
                                    atomicMax(p.qbound + t_base + qi, static_cast<unsigned long long>(mk));
                                thr[qq] = mk > thr[qq] ? mk : thr[qq];
                            }
                        }
                    }
                    // nobody appends for the next tile before the group has read the counts
                    named_bar(gbar, 128);
                }
                if (early_on && grp == 0 && !published && i + 1 == p.f_pub) early_publish();
            }
            if (early_on && grp == 0 && !published) early_publish();
        } else if (early_on) {
            // the other groups: steps A-B of the one query while the streaming groups go on
            const int etid = threadIdx.x - 64 - 128 * nstream;
            named_bar(kEarlyBar, kEpiThreads);
            if (nstream == 1)
                early_steps<kEpiThreads - 128>(p, early, 1, g, split, etid, abort_flag, &m->live_bound);
            else
                early_steps<kEpiThreads - 256>(p, early, nstream, g, split, etid, abort_flag, &m->live_bound);
        }

        // ---- final rows: every candidate of a query sorted descending, top_k kept
        uint8_t *fscr = k_smem;  // the K stages are idle once every tile has been consumed
        const uint32_t fbytes = final_scratch_bytes(p.QG, L.stage_bytes * p.kstages);
        if (FUSED) {
            // each quarter's row maxima sorted across its warp (kept in registers
            // until the K stages are free)
            unsigned long long srt[REGU ? MAXQPW : 1];
            if (REGU && !early_on && !tilepar) {
#pragma unroll
                for (int qq = 0; qq < (REGU ? MAXQPW : 1); ++qq)
                    srt[qq] = warp_sort_desc_u64(row_value(umx[qq], row), lane);
            }
            // all CTAs of the group select together (a CTA that aborted stays away,
            // and the others give up at their next group barrier)
            const bool all_ok = !named_bar_or(kEpiBar, kEpiThreads, !ok || *abort_flag != 0);
            if (all_ok && REGU && tilepar && !early_on) {
                // row maxima of the four groups' tiles combined, then sorted per quarter
                unsigned long long *comb = reinterpret_cast<unsigned long long *>(fscr + kFusedHdr + 1024);
                comb[grp * 128 + row] = umx[0];
                named_bar(kEpiBar, kEpiThreads);
                if (grp == 0) {
                    unsigned long long v = comb[row];
#pragma unroll
                    for (int g2 = 1; g2 < npar; ++g2) v = comb[g2 * 128 + row] > v ? comb[g2 * 128 + row] : v;
                    srt[0] = warp_sort_desc_u64(row_value(v, row), lane);
                }
            }
            if (all_ok) {
                const uint32_t kst = L.stage_bytes * p.kstages;
                if (early_on) {
                    // steps A-B are done: the header is in the early area, all of the K stages hold data
                    fused_tail<REGU>(buf, m->cnt, reinterpret_cast<FusedSmem *>(early),
                                     reinterpret_cast<uint64_t *>(fscr), static_cast<int>(kst / 8), p, g, split,
                                     threadIdx.x - 64, abort_flag, true);
                } else {
                    if (REGU && q_lo < q_hi) {
                        unsigned long long *sd = reinterpret_cast<unsigned long long *>(fscr + kFusedHdr);
#pragma unroll
                        for (int qq = 0; qq < (REGU ? MAXQPW : 1); ++qq)
                            if (q_lo + qq < q_hi) sd[(q_lo + qq) * 128 + row] = srt[qq];
                    }
                    fused_tail<REGU>(buf, m->cnt, reinterpret_cast<FusedSmem *>(fscr),
                                     reinterpret_cast<uint64_t *>(fscr + kFusedHdr),
                                     static_cast<int>((kst - kFusedHdr) / 8), p, g, split, threadIdx.x - 64,
                                     abort_flag, false);
                }
            }
        } else if (p.QG == 1) {
            // one query: all sixteen epilogue warps sort it together
            const bool all_ok = !named_bar_or(kEpiBar, kEpiThreads, !ok || *abort_flag != 0);
            if (all_ok && t_base < p.n_q) finish_row<16>(buf, &m->cnt[0], fscr, p, t_base, split, threadIdx.x - 64, kEpiBar);
        } else if (q_lo < q_hi && ok) {
            uint8_t *gscr = fscr + static_cast<uint32_t>(grp) * fbytes;
            for (int qi = q_lo; qi < q_hi; ++qi) {
                const long long t = t_base + qi;
                if (t >= p.n_q) break;
                finish_row<4>(buf + qi * cap, &m->cnt[qi], gscr, p, t, split, gtid, gbar);
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (FUSED && p.f_done != nullptr && threadIdx.x == 0) {
        // every CTA gets here (all waits are bounded); the group's last one has
        // seen every other CTA past all group barriers and clears the slot
        __threadfence();
        if (atomicAdd(p.f_done + g, 1u) == static_cast<unsigned>(p.splits) - 1u) {
            p.f_bar[g] = 0u;
            p.f_done[g] = 0u;
        }
    }
    // this CTA's results are written: a dependent merge grid may be scheduled
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, p.tmem_cols);
    }
}

// ------------------------------------------------------------------ merge
struct MergeParams {
    const uint64_t *part;  // [n_q][splits][top_k], each list sorted descending, 0 = empty
    int32_t *out_idx;
    float *out_score;
    long long n_q;
    int splits, top_k;
};

constexpr int kMaxSplits = 512;
constexpr int kMergeThreads = 512;
constexpr int kMergeWarps = kMergeThreads / 32;
constexpr int kMergeCap = 8192;                    // merge candidate buffer (keys)
constexpr int kMergeLevels = 5;                    // prefix lengths r0, 2 r0, ..., 16 r0
constexpr int kMergeCutR = kMergeCap / kMergeThreads;
constexpr int kMergeSortR = 2048 / kMergeThreads;  // top_k <= 2048

struct MergeMisc {
    CutScratch<8, kMergeWarps> cut;
    SortScratch<kMergeWarps> sort;
    unsigned long long bound;  // keys >= bound may be in the result
    unsigned long long lev_lo[kMergeLevels];
    unsigned long long lev_hi[kMergeLevels];
    int lev_hist[kMergeLevels * 256];
    int cnt;
};

// Merge shared memory: candidate buffer, sort scratch keys, counters.
constexpr size_t kMergeSmem = static_cast<size_t>(kMergeCap) * 8 + 2048 * 8 + sizeof(MergeMisc);

// Merge of the sorted per-split top-k lists of one query (one CTA per query)
// into its output row.
//
// 1. A lower bound on the final top_k-th key: for a prefix length r, if
//    c = ceil(top_k / r) lists have their r-th key >= v, then at least top_k
//    real keys are >= v, so the c-th largest of the lists' r-th keys is a
//    bound; so is anything below it, e.g. the lower edge of the histogram bin
//    that holds it. It is computed for r = r0, 2 r0, ..., 16 r0 (r0 the
//    shortest prefix with c <= splits) from one histogram per level; the
//    largest bound wins. (Several lengths matter when most lists hold only
//    masked keys for this query.)
// 2. Each list contributes its prefix of keys >= the bound (the lists are
//    sorted): each warp reads the heads of its lists, 32 keys at a time, all
//    loads in flight together, and appends the passing keys to the buffer.
// 3. The candidates are cut to top_k if there are too many to sort at once,
//    sorted, and written.
__global__ void __launch_bounds__(kMergeThreads, 1) merge_kernel(const MergeParams p) {
    extern __shared__ uint8_t smem_raw[];
    uint64_t *buf = reinterpret_cast<uint64_t *>(smem_raw);
    uint64_t *tmp = buf + kMergeCap;
    MergeMisc *m = reinterpret_cast<MergeMisc *>(smem_raw + static_cast<size_t>(kMergeCap + 2048) * 8);
    constexpr int T = kMergeThreads;
    const int tid = threadIdx.x;
    const int lane = tid & 31;
    const int warp = tid >> 5;
    const long long t = blockIdx.x;
    const int S = p.splits;
    const int K = p.top_k;
    const uint64_t *lists = p.part + t * static_cast<long long>(S) * K;
    // launched as a programmatic dependent of the scoring kernel: everything
    // above overlaps its tail; its results are read only after this wait
    asm volatile("griddepcontrol.wait;" ::: "memory");

    if (S * K <= kMergeCap) {
        // ---- 1-2 for lists that fit the buffer together: every real key is
        // appended at once (one round of loads; no bound, no walk along the lists)
        if (tid == 0) m->cnt = 0;
        named_bar(1, T);
        constexpr int U = kMergeCap / T;
        uint64_t v[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int i = tid + u * T;
            v[u] = i < S * K ? lists[i] : 0ull;
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            if (u * T < S * K) warp_append(buf, &m->cnt, v[u], v[u] != 0ull, lane);  // 0: no key
        }
        named_bar(1, T);
    } else {
        // ---- 1. bound
        int r0 = 1;
        while ((K + r0 - 1) / r0 > S) r0 <<= 1;
        int nlev = 0;
        while (nlev < kMergeLevels && (r0 << nlev) <= K) ++nlev;
        uint64_t *vals = buf;  // [level][list]: the lists' r-th keys (0 where a list is shorter)
        {
            constexpr int U = kMergeLevels * kMaxSplits / T;  // loads per thread at most, all in flight
            uint64_t v[U];
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int i = tid + u * T;
                v[u] = 0ull;
                if (i < nlev * S) {
                    const int lev = i / S, j = i - lev * S;
                    v[u] = lists[static_cast<long long>(j) * K + (r0 << lev) - 1];
                }
            }
#pragma unroll
            for (int u = 0; u < U; ++u)
                if (tid + u * T < nlev * S) vals[tid + u * T] = v[u];
        }
        if (tid == 0) {
            m->bound = 0ull;
            m->cnt = 0;
        }
        named_bar(1, T);
        // per level: the smallest and largest nonzero value, then one 8-bit histogram
        // of the digit just below their common bits. The lower edge of the bin that
        // holds rank c is <= the c-th largest value, so at least c lists have their
        // r-th key at or above it: a (slightly looser) bound without a full select.
        {
            unsigned long long lo = ~0ull, hi = 0ull;
            const int lev = warp < nlev ? warp : 0;
            if (warp < nlev) {
                for (int j = lane; j < S; j += 32) {
                    const unsigned long long v = vals[lev * S + j];
                    if (v != 0ull) {
                        lo = v < lo ? v : lo;
                        hi = v > hi ? v : hi;
                    }
                }
                lo = warp_min_u64(lo);
                hi = warp_max_u64(hi);
                if (lane == 0) {
                    m->lev_lo[lev] = lo;
                    m->lev_hi[lev] = hi;
                }
            }
            for (int i = tid; i < kMergeLevels * 256; i += T) m->lev_hist[i] = 0;
            named_bar(1, T);
            for (int task = tid; task < nlev * S; task += T) {
                const int l = task / S;
                const uint64_t v = vals[task];
                const uint64_t a = m->lev_lo[l], b = m->lev_hi[l];
                if (v == 0ull || a == ~0ull) continue;
                const uint64_t diff = a ^ b;
                const int hb = diff ? 63 - __clzll(static_cast<long long>(diff)) : 0;
                atomicAdd(&m->lev_hist[l * 256 + key_digit<8>(v, hb - 7)], 1);
            }
            named_bar(1, T);
            if (warp < nlev) {
                const uint64_t a = m->lev_lo[lev], b = m->lev_hi[lev];
                const int c = (K + (r0 << lev) - 1) / (r0 << lev);
                int total = 0;
                for (int i = lane; i < 256; i += 32) total += m->lev_hist[lev * 256 + i];
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) total += __shfl_xor_sync(0xFFFFFFFFu, total, o);
                if (a != ~0ull && total >= c) {
                    int d, above, inbin;
                    scan_digit<8>(m->lev_hist + lev * 256, c, lane, d, above, inbin);
                    const uint64_t diff = a ^ b;
                    const int hb = diff ? 63 - __clzll(static_cast<long long>(diff)) : 0;
                    const int shift = hb - 7;
                    const uint64_t keep = hb >= 63 ? 0ull : ~((2ull << hb) - 1ull);  // bits all values share
                    uint64_t edge = (a & keep) | digit_bits(d, shift);
                    if (edge == 0ull) edge = 1ull;
                    if (lane == 0) atomicMax(&m->bound, edge);
                }
            }
        }
        named_bar(1, T);
        const unsigned long long thr = m->bound ? m->bound - 1ull : 0ull;  // keys > thr pass
        named_bar(1, T);  // everyone has read the bound; buf is free again

        // ---- 2. surviving prefixes into the buffer. Warp w owns lists w + 16 u;
        // per step it reads 32 keys of 8 of them (loads in flight together), so a
        // step of the block appends at most 32 * 128 keys.
        uint64_t run = thr;  // running threshold of the buffer (uniform)
        const int owned = (S - warp + kMergeWarps - 1) / kMergeWarps;  // lists of this warp (<= 32)
        uint32_t active = owned >= 32 ? 0xFFFFFFFFu : ((1u << owned) - 1u);
        const int nbatch = ((S + kMergeWarps - 1) / kMergeWarps + 7) / 8;  // uniform
        for (int base = 0; base < K; base += 32) {
            for (int b = 0; b < nbatch; ++b) {
                uint64_t key[8];
#pragma unroll
                for (int u8 = 0; u8 < 8; ++u8) {
                    const int u = b * 8 + u8;
                    const int j = warp + kMergeWarps * u;
                    const bool on = u < 32 && ((active >> u) & 1u) && base + lane < K;
                    key[u8] = on ? lists[static_cast<long long>(j) * K + base + lane] : 0ull;
                }
#pragma unroll
                for (int u8 = 0; u8 < 8; ++u8) {
                    const int u = b * 8 + u8;
                    if (u < 32 && ((active >> u) & 1u)) {
                        const bool pass = key[u8] > run;
                        const unsigned bal = __ballot_sync(0xFFFFFFFFu, pass);
                        if (bal != 0xFFFFFFFFu) active &= ~(1u << u);  // the list's prefix ends here
                        warp_append(buf, &m->cnt, key[u8], pass, lane);
                    }
                }
                named_bar(1, T);
                const int n = m->cnt;
                named_bar(1, T);  // every thread has read cnt before anyone changes it
                if (n > kMergeCap - 32 * 8 * kMergeWarps) {
                    uint64_t mk;
                    group_cut<kMergeCutR, 8, kMergeWarps>(buf, &m->cnt, n, K, 64, false, tid, 1, &m->cut, &mk);
                    run = mk;
                }
            }
            if (!named_bar_or(1, T, active != 0u)) break;
        }
    }

    // ---- 3. cut, sort, write
    int n = m->cnt;
    if (n > 2048) {
        uint64_t mk;
        group_cut<kMergeCutR, 8, kMergeWarps>(buf, &m->cnt, n, K, 0, true, tid, 1, &m->cut, &mk);
        n = K;
    }
    group_sort_desc<kMergeSortR, kMergeWarps>(buf, tmp, n, tid, 1, &m->sort);
    for (int j = tid; j < K; j += T) {
        int32_t idx;
        float sc;
        decode_key(j < n ? buf[j] : 0ull, idx, sc);
        p.out_idx[t * K + j] = idx;
        p.out_score[t * K + j] = sc;
    }
}

// Merge of a few sorted per-split lists (splits <= kRankMaxSplits, splits *
// top_k <= kRankMaxKeys), one CTA per query: a key's place in the output is
// the number of larger keys over all lists (keys are unique), i.e. its
// position in its own list plus, for every other list, a binary search for
// where it would go. The keys of rank < top_k land in their output slots; the
// slots past the number of real keys get (-1, -inf). No barrier after the
// lists are staged, no radix passes: a short CTA, several per SM.
constexpr int kRankThreads = 256;
constexpr int kRankMaxSplits = 8;
constexpr int kRankMaxKeys = 4096;

__global__ void __launch_bounds__(kRankThreads) merge_ranked_kernel(const MergeParams p) {
    extern __shared__ uint8_t smem_raw[];
    uint64_t *keys = reinterpret_cast<uint64_t *>(smem_raw);  // [splits][top_k]
    __shared__ int len[kRankMaxSplits];                       // real keys per list
    const int S = p.splits, K = p.top_k, SK = S * K;
    const long long t = blockIdx.x;
    const uint64_t *lists = p.part + t * static_cast<long long>(SK);
    asm volatile("griddepcontrol.wait;" ::: "memory");  // the scoring grid's lists are complete
    for (int i = threadIdx.x; i < SK; i += kRankThreads) keys[i] = lists[i];
    __syncthreads();
    if (threadIdx.x < S) {
        // sorted descending with 0 (no key) at the end: the first 0 is the length
        const uint64_t *l = keys + threadIdx.x * K;
        int lo = 0, hi = K;
        while (lo < hi) {
            const int mid = (lo + hi) >> 1;
            if (l[mid] != 0ull) lo = mid + 1;
            else hi = mid;
        }
        len[threadIdx.x] = lo;
    }
    __syncthreads();
    int total = 0;
    for (int j = 0; j < S; ++j) total += len[j];
    int32_t *oi = p.out_idx + t * K;
    float *os = p.out_score + t * K;
    for (int i = threadIdx.x; i < SK; i += kRankThreads) {
        const int j = i / K, pos = i - j * K;
        if (pos >= len[j]) continue;
        const uint64_t x = keys[i];
        // (the search stops once the count reaches top_k: most keys of the lists
        // are not in the output and drop out after a list or two)
        int rank = pos;
        for (int j2 = 0; j2 < S && rank < K; ++j2) {
            if (j2 == j) continue;
            const uint64_t *l = keys + j2 * K;
            int lo = 0, hi = len[j2];  // keys of list j2 larger than x: the first index whose key is below x
            while (lo < hi) {
                const int mid = (lo + hi) >> 1;
                if (l[mid] > x) lo = mid + 1;
                else hi = mid;
            }
            rank += lo;
        }
        if (rank < K) {
            int32_t idx;
            float sc;
            decode_key(x, idx, sc);
            oi[rank] = idx;
            os[rank] = sc;
        }
    }
    for (int r = total + threadIdx.x; r < K; r += kRankThreads) {
        oi[r] = -1;
        os[r] = __uint_as_float(0xFF800000u);
    }
}

// Rows of (-1, -inf): the whole output when there are no keys.
__global__ void fill_empty_kernel(int32_t *out_idx, float *out_score, long long n) {
    for (long long i = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; i < n;
         i += static_cast<long long>(gridDim.x) * blockDim.x) {
        out_idx[i] = -1;
        out_score[i] = __uint_as_float(0xFF800000u);
    }
}

}  // namespace lid
