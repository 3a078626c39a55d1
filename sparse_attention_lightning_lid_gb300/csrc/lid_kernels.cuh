// lid_kernels.cuh -- the lightning-indexer scoring + streaming top-k kernel
// and the split merge kernel, sm_103a.
//
// Per CTA: one group of QG queries (QG*H rows of q, the MMA's N) and one
// contiguous range of 128-key tiles (a split). Warp roles:
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
//               final sorts run side by side.
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
constexpr int kSortMax = 2048;  // keys a final sort takes at once (more are first cut to top_k)
constexpr int kCutDB = 6;       // digit bits of the streaming cuts
constexpr int kSortScratchBytes = (static_cast<int>(sizeof(SortScratch<16>)) + 63) & ~63;
constexpr int kCutScratchBytes = (static_cast<int>(sizeof(CutScratch<8, 16>)) + 63) & ~63;
// final-phase scratch one sorter needs (counters + kSortMax keys)
constexpr int kFinalScratchBytes = kSortScratchBytes + kCutScratchBytes + kSortMax * 8;

struct ScoreParams {
    const uint16_t *mask;  // [n_q][n_kv] f16 bits or null
    const float *w;        // [n_q][H]
    int32_t *out_idx;      // [n_q][top_k] (splits == 1)
    float *out_score;
    uint64_t *part;        // [n_q][splits][top_k] sorted keys (splits > 1)
    int *tickets;          // [n_q] zeroed here for the merge (splits > 1)
    long long n_q, n_kv;
    int D, QG, N, top_k, P;  // P = top_k rounded up to a power of two
    int n_groups, splits, tiles_per_split, n_tiles;
    int kstages, acc_stages, cap, tmem_cols;
    uint32_t idesc;
};

struct Misc {
    uint64_t k_full[kMaxKStages];
    uint64_t k_empty[kMaxKStages];
    uint64_t acc_full[kMaxAccStages];
    uint64_t acc_empty[kMaxAccStages];
    uint64_t q_full;
    int cnt[kMaxQG];
    CutScratch<kCutDB, 4> cut[kEPG];
    uint32_t tmem_base;
    int abort_flag;
};

struct SmemLayout {
    uint32_t stage_bytes, k_off, q_off, w_off, buf_off, misc_off, total;
};

// Offsets from a 1024-byte aligned base; `total` includes the alignment slack.
__host__ __device__ inline SmemLayout smem_layout(int D, int N, int QG, int H, int kstages, int cap) {
    SmemLayout L;
    L.stage_bytes = static_cast<uint32_t>(kBM * D * 2);
    L.k_off = 0;
    L.q_off = L.k_off + L.stage_bytes * kstages;
    L.w_off = L.q_off + static_cast<uint32_t>(N * D * 2);
    L.buf_off = L.w_off + ((static_cast<uint32_t>(QG * H * 4) + 15u) & ~15u);
    L.misc_off = L.buf_off + static_cast<uint32_t>(QG) * static_cast<uint32_t>(cap) * 8u;
    L.total = L.misc_off + ((static_cast<uint32_t>(sizeof(Misc)) + 15u) & ~15u) + 1024u;
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

__device__ __forceinline__ float f16_bits_to_float(uint16_t b) {
    return __half2float(__ushort_as_half(b));
}

// Sort the n candidate keys of row t and write the top_k: the final output
// row (splits == 1) or this split's sorted list. More than kSortMax keys are
// first cut to exactly top_k. `scratch` holds the cut's and the sort's
// counters followed by kSortMax keys of temporary space.
template <int NW>
__device__ void finish_row(uint64_t *b, int *cnt, uint8_t *scratch, const ScoreParams &p, long long t, int split,
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
        if (split == 0 && tid == 0) p.tickets[t] = 0;
    }
    named_bar(bar, T);
}

template <int H>
__global__ void __maxnreg__(96)
    score_select_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_q,
                        const ScoreParams p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const SmemLayout L = smem_layout(p.D, p.N, p.QG, H, p.kstages, p.cap);
    uint8_t *k_smem = smem + L.k_off;
    uint8_t *q_smem = smem + L.q_off;
    float *w_s = reinterpret_cast<float *>(smem + L.w_off);
    uint64_t *buf = reinterpret_cast<uint64_t *>(smem + L.buf_off);
    Misc *m = reinterpret_cast<Misc *>(smem + L.misc_off);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int g = blockIdx.x % p.n_groups;
    const int split = blockIdx.x / p.n_groups;
    const int tile0 = split * p.tiles_per_split;
    const int tile1 = min(tile0 + p.tiles_per_split, p.n_tiles);
    const int ntl = max(0, tile1 - tile0);
    constexpr int ne_threads = kEpiThreads;
    const long long t_base = static_cast<long long>(g) * p.QG;

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
        m->abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc(&m->tmem_base, p.tmem_cols);
        tmem_relinquish();
    }
    if (warp >= 2) {
        const int etid = threadIdx.x - 64;
        for (int i = etid; i < p.QG * H; i += ne_threads) {
            const long long t = t_base + i / H;
            w_s[i] = (t < p.n_q) ? p.w[t * H + (i % H)] : 0.f;
        }
        for (int i = etid; i < p.QG; i += ne_threads) m->cnt[i] = 0;
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = m->tmem_base;
    volatile int *abort_flag = &m->abort_flag;

    if (warp == 0) {
        // ------------------------------------------------------ TMA producer
        if (lane == 0) {
            tma_prefetch_desc(&tm_k);
            tma_prefetch_desc(&tm_q);
            const int nchunk = p.D / 64;
            if (ntl > 0) {
                mbar_arrive_expect_tx(&m->q_full, static_cast<uint32_t>(p.N * p.D * 2));
                for (int c = 0; c < nchunk; ++c)
                    tma_load_2d(q_smem + c * p.N * 128, &tm_q, c * 64, static_cast<int>(t_base * H),
                                &m->q_full);
            }
            int issued = 0;
            for (int i = 0; i < ntl; ++i) {
                const int s = i % p.kstages;
                const uint32_t ph = static_cast<uint32_t>(i / p.kstages) & 1u;
                if (i >= p.kstages && !mbar_wait(&m->k_empty[s], ph ^ 1u, abort_flag, 1)) break;
                mbar_arrive_expect_tx(&m->k_full[s], L.stage_bytes);
                uint8_t *dst = k_smem + s * L.stage_bytes;
                for (int c = 0; c < nchunk; ++c)
                    tma_load_2d(dst + c * kBM * 128, &tm_k, c * 64, (tile0 + i) * kBM, &m->k_full[s]);
                issued = i + 1;
            }
            // wait (bounded) for loads still in flight before the CTA may exit
            const int first = max(0, issued - p.kstages);
            for (int i = first; i < issued; ++i) {
                const int s = i % p.kstages;
                const uint32_t ph = static_cast<uint32_t>(i / p.kstages) & 1u;
                int dummy = 0;
                mbar_wait(&m->k_full[s], ph, &dummy, 1);
            }
            if (ntl > 0) {
                int dummy = 0;
                mbar_wait(&m->q_full, 0, &dummy, 1);
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        // ------------------------------------------------------- MMA issuer
        if (lane == 0) {
            const uint32_t q_addr = smem_u32(q_smem);
            const uint32_t k_addr = smem_u32(k_smem);
            bool ok = ntl == 0 || mbar_wait(&m->q_full, 0, abort_flag, 2);
            tc_fence_after();
            for (int i = 0; ok && i < ntl; ++i) {
                const int s = i % p.kstages;
                const uint32_t kph = static_cast<uint32_t>(i / p.kstages) & 1u;
                const int a = i % p.acc_stages;
                const uint32_t aph = static_cast<uint32_t>(i / p.acc_stages) & 1u;
                if (!mbar_wait(&m->k_full[s], kph, abort_flag, 2)) break;
                if (i >= p.acc_stages && !mbar_wait(&m->acc_empty[a], aph ^ 1u, abort_flag, 2)) break;
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(a * p.N);
                const uint32_t ks = k_addr + s * L.stage_bytes;
                for (int kk = 0; kk < p.D / 16; ++kk) {
                    const uint32_t off = static_cast<uint32_t>((kk & 3) * 32);
                    const uint64_t adesc = smem_desc_sw128(ks + (kk >> 2) * kBM * 128 + off);
                    const uint64_t bdesc = smem_desc_sw128(q_addr + (kk >> 2) * p.N * 128 + off);
                    umma_f16(d_tmem, adesc, bdesc, p.idesc, kk > 0 ? 1u : 0u);
                }
                umma_commit(&m->k_empty[s]);
                umma_commit(&m->acc_full[a]);
            }
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
        constexpr int LW = H < 32 ? H : 32;            // columns per TMEM load
        constexpr int MAXQPW = H >= 64 ? 1 : 64 / H;   // queries per group at most
        constexpr int CUT_R = kSortMax / 128;          // keys per thread a group cut holds in registers
        CutScratch<kCutDB, 4> *cs = &m->cut[grp];
        // running threshold of each of my queries (keys above it are candidates)
        uint64_t thr[MAXQPW];
#pragma unroll
        for (int qq = 0; qq < MAXQPW; ++qq) thr[qq] = 0ull;
        bool ok = true;

        if (q_lo < q_hi) {
            // mask values of my queries, loaded two tiles before they are used
            auto load_mask = [&](int i, float *mv) {
                const long long s = static_cast<long long>(tile0 + i) * kBM + row;
#pragma unroll
                for (int qq = 0; qq < MAXQPW; ++qq) {
                    const long long t = t_base + q_lo + qq;
                    mv[qq] = 0.f;
                    if (i < ntl && q_lo + qq < q_hi && p.mask != nullptr && t < p.n_q && s < p.n_kv)
                        mv[qq] = f16_bits_to_float(__ldg(p.mask + t * p.n_kv + s));
                }
            };
            float mval[MAXQPW], mnext[MAXQPW];
            load_mask(0, mval);
            load_mask(1, mnext);
            for (int i = 0; i < ntl; ++i) {
                const int a = i % p.acc_stages;
                const uint32_t aph = static_cast<uint32_t>(i / p.acc_stages) & 1u;
                const long long s = static_cast<long long>(tile0 + i) * kBM + row;
                const bool s_ok = s < p.n_kv;
                float mlater[MAXQPW];
                load_mask(i + 2, mlater);
                ok = mbar_wait(&m->acc_full[a], aph, abort_flag, 3);
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
                            // sum_h w[h] * relu(S[h]) on packed pairs of heads, two chains,
                            // LW accumulator columns at a time
                            const float4 *w4 = reinterpret_cast<const float4 *>(w_s + qi * H);
                            uint64_t acc0 = 0ull, acc1 = 0ull;
#pragma unroll
                            for (int c = 0; c < H; c += LW) {
                                uint32_t x[LW];
                                tmem_ld<LW>(tacc + qi * H + c, x);
                                tmem_wait_ld();
#pragma unroll
                                for (int h = 0; h < LW; h += 4) {
                                    const float4 wv = w4[(c + h) / 4];
                                    const uint64_t r01 = pack_f32x2(fmaxf(__uint_as_float(x[h]), 0.f),
                                                                    fmaxf(__uint_as_float(x[h + 1]), 0.f));
                                    const uint64_t r23 = pack_f32x2(fmaxf(__uint_as_float(x[h + 2]), 0.f),
                                                                    fmaxf(__uint_as_float(x[h + 3]), 0.f));
                                    acc0 = fma_f32x2(pack_f32x2(wv.x, wv.y), r01, acc0);
                                    acc1 = fma_f32x2(pack_f32x2(wv.z, wv.w), r23, acc1);
                                }
                            }
                            const long long t = t_base + qi;
                            const float score = (sum_f32x2(acc0) + sum_f32x2(acc1)) + mval[qq];
                            const bool valid = s_ok && t < p.n_q;
                            const uint64_t key = valid ? make_key(score, static_cast<uint32_t>(s)) : 0ull;
                            const int after =
                                warp_append(buf + qi * cap, &m->cnt[qi], key, valid && key > thr[qq], lane);
                            // the last warp to append sees the final count, so this vote is exact
                            overflow |= after > cap - kBM;
                        }
                    }
                }
#pragma unroll
                for (int qq = 0; qq < MAXQPW; ++qq) {
                    mval[qq] = mnext[qq];
                    mnext[qq] = mlater[qq];
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&m->acc_empty[a]);
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
                                thr[qq] = mk;
                            }
                        }
                    }
                    // nobody appends for the next tile before the group has read the counts
                    named_bar(gbar, 128);
                }
            }
        }

        // ---- final rows: every candidate of a query sorted descending, top_k kept
        uint8_t *fscr = k_smem;  // the K stages are idle once every tile has been consumed
        const uint32_t fbytes = final_scratch_bytes(p.QG, L.stage_bytes * p.kstages);
        if (p.QG == 1) {
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
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, p.tmem_cols);
    }
}

// ------------------------------------------------------------------ merge
struct MergeParams {
    const uint64_t *part;  // [n_q][splits][top_k], each list sorted descending, 0 = empty
    int *counts;           // [n_q][splits] keys of each list that pass the bound
    int *tickets;          // [n_q] finished-CTA tickets (zeroed by the scoring kernel)
    int32_t *out_idx;
    float *out_score;
    long long n_q;
    int splits, top_k, P, cap, lists_per_cta, ctas_per_q;
};

constexpr int kMaxSplits = 512;
constexpr int kMergeThreads = 512;
constexpr int kMergeCap = 8192;                   // merge candidate buffer (keys)
constexpr int kMergeCutR = kMergeCap / kMergeThreads;
constexpr int kMergeSortR = 2048 / kMergeThreads;  // top_k <= 2048

struct MergeMisc {
    CutScratch<8, kMergeThreads / 32> cut;
    SortScratch<kMergeThreads / 32> sort;
    unsigned long long bound;  // keys >= bound may be in the result
    int cnt;
    int last;
    int pre[kMaxSplits + 1];   // prefix sums of the per-list counts
};

// Merge shared memory: candidate buffer, sort scratch keys, counters.
constexpr size_t kMergeSmem = static_cast<size_t>(kMergeCap) * 8 + 2048 * 8 + sizeof(MergeMisc);

// Final top_k of buf[0, m->cnt), sorted, decoded into the output row t.
__device__ void merge_finish(uint64_t *buf, uint64_t *tmp, const MergeParams &p, MergeMisc *m, long long t,
                             int tid, int T) {
    int n = m->cnt;
    if (n > 2048) {
        uint64_t mk;
        group_cut<kMergeCutR, 8, kMergeThreads / 32>(buf, &m->cnt, n, p.top_k, 0, true, tid, 1, &m->cut, &mk);
        n = p.top_k;
    }
    group_sort_desc<kMergeSortR, kMergeThreads / 32>(buf, tmp, n, tid, 1, &m->sort);
    for (int j = tid; j < p.top_k; j += T) {
        int32_t idx;
        float sc;
        decode_key(j < n ? buf[j] : 0ull, idx, sc);
        p.out_idx[t * p.top_k + j] = idx;
        p.out_score[t * p.top_k + j] = sc;
    }
}

// Merge of the sorted per-split top-k lists of each query into its row.
//
// 1. A lower bound on the final top_k-th key: for a prefix length r, if c =
//    ceil(top_k / r) lists have their r-th key >= v, then at least top_k real
//    keys are >= v; so the c-th largest of the lists' r-th keys is a bound.
//    One warp per r in {1, 2, 4, ...} computes it by counting; the largest wins.
// 2. Each list contributes only its prefix of keys >= the bound (the lists
//    are sorted): one warp per list reads 32 keys at a time until one fails.
// 3. The CTA that finishes last for the query (atomic ticket after a fence;
//    nothing waits) streams all surviving prefixes through a running top-k,
//    sorts the result and writes the row.
// Grid: n_q * ctas_per_q CTAs; CTA mc of a query handles lists
// [mc * lists_per_cta, (mc + 1) * lists_per_cta).
__global__ void __launch_bounds__(kMergeThreads, 1) merge_kernel(const MergeParams p) {
    extern __shared__ uint8_t smem_raw[];
    uint64_t *buf = reinterpret_cast<uint64_t *>(smem_raw);
    uint64_t *tmp = buf + kMergeCap;
    MergeMisc *m = reinterpret_cast<MergeMisc *>(smem_raw + static_cast<size_t>(kMergeCap + 2048) * 8);
    const int tid = threadIdx.x;
    const int T = blockDim.x;
    const int lane = tid & 31;
    const int warp = tid >> 5;
    const int nwarps = T >> 5;
    const long long t = blockIdx.x / p.ctas_per_q;
    const int mc = blockIdx.x % p.ctas_per_q;
    const int S = p.splits;
    const uint64_t *lists = p.part + t * static_cast<long long>(S) * p.top_k;
    if (tid == 0) {
        m->bound = 0ull;
        m->cnt = 0;
    }
    named_bar(1, T);
    // ---- 1. bound
    {
        const int r = 1 << warp;
        const int c = (p.top_k + r - 1) / r;
        if (r <= p.top_k && c <= S) {
            uint64_t *vals = buf + warp * kMaxSplits;  // staging, S <= kMaxSplits
            for (int j = lane; j < S; j += 32) vals[j] = lists[static_cast<long long>(j) * p.top_k + r - 1];
            __syncwarp();
            unsigned long long best = 0ull;
            for (int j = lane; j < S; j += 32) {
                const uint64_t v = vals[j];
                if (v == 0ull) continue;
                int greater = 0;
                for (int i = 0; i < S; ++i) greater += vals[i] > v;
                if (greater == c - 1) best = v;
            }
            best = warp_max_u64(best);
            if (lane == 0 && best != 0ull) atomicMax(&m->bound, best);
        }
    }
    named_bar(1, T);
    const unsigned long long thr = m->bound ? m->bound - 1ull : 0ull;  // keys > thr pass
    // ---- 2. surviving prefix length of each of my lists
    const int l0 = mc * p.lists_per_cta;
    const int l1 = min(S, l0 + p.lists_per_cta);
    for (int j = l0 + warp; j < l1; j += nwarps) {
        const uint64_t *L = lists + static_cast<long long>(j) * p.top_k;
        int c = 0;
        for (int base = 0; base < p.top_k; base += 32) {
            const int i = base + lane;
            const bool pass = i < p.top_k && L[i] > thr;
            const unsigned bal = __ballot_sync(0xFFFFFFFFu, pass);
            c += __popc(bal);
            if (bal != 0xFFFFFFFFu) break;
        }
        if (lane == 0) p.counts[t * S + j] = c;
    }
    if (p.ctas_per_q > 1) {
        __threadfence();
        named_bar(1, T);
        if (tid == 0) m->last = atomicAdd(p.tickets + t, 1) == p.ctas_per_q - 1;
        named_bar(1, T);
        if (!m->last) return;
        __threadfence();
    } else {
        named_bar(1, T);
    }
    // ---- 3. stream the surviving prefixes
    if (warp == 0) {
        // exclusive prefix sums of the counts; lane l owns a run of ceil(S/32) lists
        const int per = (S + 31) / 32;
        const int j0 = lane * per;
        int run = 0;
        for (int j = j0; j < min(S, j0 + per); ++j)
            run += *reinterpret_cast<volatile int *>(p.counts + t * S + j);
        int incl = run;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int v = __shfl_up_sync(0xFFFFFFFFu, incl, o);
            if (lane >= o) incl += v;
        }
        int acc = incl - run;
        for (int j = j0; j < min(S, j0 + per); ++j) {
            m->pre[j] = acc;
            acc += *reinterpret_cast<volatile int *>(p.counts + t * S + j);
        }
        if (lane == 31) m->pre[S] = incl;
    }
    named_bar(1, T);
    const int total = m->pre[S];
    uint64_t thr_run = 0ull;  // running threshold of the stream (uniform)
    for (int base = 0; base < total; base += T) {
        const int i = base + tid;
        uint64_t key = 0ull;
        if (i < total) {
            int lo = 0, hi = S;  // largest j with pre[j] <= i
            while (hi - lo > 1) {
                const int mid = (lo + hi) >> 1;
                if (m->pre[mid] <= i) lo = mid; else hi = mid;
            }
            key = lists[static_cast<long long>(lo) * p.top_k + (i - m->pre[lo])];
        }
        warp_append(buf, &m->cnt, key, key > thr_run, lane);
        named_bar(1, T);
        const int n = m->cnt;
        named_bar(1, T);  // every thread has read cnt before anyone changes it
        if (n > kMergeCap - T) {
            uint64_t mk;
            group_cut<kMergeCutR, 8, kMergeThreads / 32>(buf, &m->cnt, n, p.top_k, 64, false, tid, 1, &m->cut, &mk);
            thr_run = mk;
        }
    }
    merge_finish(buf, tmp, p, m, t, tid, T);
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
