// lid_stream.cuh -- the single-query kernel, sm_103a: one query row per CTA,
// the row's keys split over up to one CTA per SM (the decode shape), merged
// inside the same cooperative launch.
//
// It computes what score_select_kernel computes for such a call, with a small
// code body so that the once-per-launch steps do not wait on instruction
// fetch. Warp roles (448 threads):
//   warp 0       TMA: q once, then the CTA's K tiles into a ring of stages
//   warp 1       tensor memory and tcgen05.mma: S = K_tile . Q^T (keys on M,
//                heads on N) into one of four accumulators
//   warps 2-9    two streaming groups taking the tiles in turn: per key (one
//                TMEM lane per thread) sum_h w[h] relu(S[h]) + mask, the key
//                into the CTA's candidate buffer if it is not below the
//                certified bound (once that is known), and its row maximum
//   warps 10-13  merge group: after f_pub tiles it takes the streaming groups'
//                row maxima, publishes the CTA's certificates, meets the other
//                CTAs of the row once, and derives the certified bound B
// Tail (all 384 epilogue threads): the CTA's keys >= B go to its fixed region
// (plain stores), the CTAs meet a second time, each loads every region,
// packs the candidates in the same order and ranks its slice of them. A CTA
// with more keys >= B than its region holds also writes them (at most top_k,
// its own top ones) to an overflow list that every CTA then adds.
#pragma once

#include "lid_kernels.cuh"

namespace lid {

constexpr int kSQThreads = 448;
constexpr int kSQEpi = 384;     // epilogue threads: two streaming groups and the merge group
constexpr int kSQAcc = 4;       // accumulator stages in tensor memory
constexpr int kSQRegion = 32;   // region slots per split: the count, then up to 31 keys
constexpr int kSQBarPub = 1;    // streaming groups arrive with their row maxima; the merge group waits
constexpr int kSQBarM = 2;      // the merge group
constexpr int kSQBarTail = 3;   // every epilogue thread

struct SQHdr {
    uint64_t k_full[kMaxKStages], k_empty[kMaxKStages], acc_full[kSQAcc], acc_empty[kSQAcc];
    uint64_t q_full, mma_done, never;  // never: a barrier nothing arrives at (the fault-injection test)
    uint64_t side_full;                // the CTA's mask bits and key scales are in shared memory
    uint32_t tmem_base;
    int abort_flag, cnt, tile0, ntl, ovf_off;
    int m_staged, k_staged;  // keys of the CTA whose mask bits / key scales are in shared memory
    int done_counted;        // this CTA counted itself in f_done after the second meeting
    unsigned long long live_bound, bound, kth;
    int wtot[32];
    int hist[256];
    int bhist[4][256];  // the merge warps' bins of the bound step
    int bmin[4][256];   // ... and each bin's smallest value
    unsigned long long comb[2][128];  // the streaming groups' row maxima at publication
    unsigned long long srt[128];      // the combined row maxima, each quarter sorted descending
};

struct SQLayout {
    uint32_t hdr, stage, k_off, q_off, w_off, buf_off, mask_off, ks_off, total;
};

// Offsets from a 1024-byte aligned base (the K stages and q are 1024-aligned
// for the 128-byte swizzle); `total` includes the alignment slack.
__host__ __device__ inline SQLayout sq_layout(int D, int H, int esize, int kstages, int cap) {
    SQLayout L;
    L.hdr = (static_cast<uint32_t>(sizeof(SQHdr)) + 1023u) & ~1023u;
    L.stage = static_cast<uint32_t>(kBM * D * esize);
    L.k_off = L.hdr;
    L.q_off = L.k_off + L.stage * static_cast<uint32_t>(kstages);
    L.w_off = L.q_off + static_cast<uint32_t>(H * D * esize);
    L.buf_off = L.w_off + ((static_cast<uint32_t>(H) * 4u + 15u) & ~15u);
    L.mask_off = L.buf_off + static_cast<uint32_t>(cap) * 8u;  // the CTA's mask bits: [cap] f16
    L.ks_off = L.mask_off + ((static_cast<uint32_t>(cap) * 2u + 15u) & ~15u);  // its key scales: [cap] f32
    L.total = L.ks_off + static_cast<uint32_t>(cap) * 4u + 1024u;
    return L;
}

// Group barrier of the launch's CTAs of query group g (one thread per CTA):
// arrive, then wait (bounded) until `target` arrivals. False on a timeout.
__device__ __forceinline__ bool sq_grid_wait(const ScoreParams &p, int g, unsigned target, volatile int *abort_flag) {
    unsigned *ctr = p.f_bar + g;
    asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(ctr), "r"(1u) : "memory");
    if (ld_acquire_u32(ctr) >= target) return true;
    const long long t0 = clock64();
    while (ld_acquire_u32(ctr) < target) {
        if (clock64() - t0 > p.wait_limit) {
            *abort_flag = 1;
            atomicCAS(&g_dev_error, 0, 4);
            return false;
        }
    }
    return true;
}

// sum_h w[h] * relu(S[h]) of one key (this thread's TMEM lane), from the
// accumulator columns at tacc, loads of the next 16 columns in flight while
// the current ones are summed; half the heads as (w x + w |x|) / 2 on the FMA
// pipe, the other half with max on the ALU pipe.
template <int H>
__device__ __forceinline__ float sq_head_sum(uint32_t tacc, const float *w_s) {
    const float4 *w4 = reinterpret_cast<const float4 *>(w_s);
    uint64_t acc0 = 0ull, acc1 = 0ull, accx = 0ull;
    float acca0 = 0.f, acca1 = 0.f;
    constexpr int CW = 16;
    uint32_t xa[CW], xb[CW];
    tmem_ld<CW>(tacc, xa);
    tmem_wait_ld_dep<CW>(xa);
#pragma unroll
    for (int c = 0; c < H; c += CW) {
        uint32_t *cur = ((c / CW) & 1) ? xb : xa;
        uint32_t *nxt = ((c / CW) & 1) ? xa : xb;
        if (c + CW < H) tmem_ld<CW>(tacc + c + CW, nxt);
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
        if (c + CW < H) tmem_wait_ld_dep<CW>(nxt);
    }
    return (sum_f32x2(acc0) + sum_f32x2(acc1)) + 0.5f * (sum_f32x2(accx) + (acca0 + acca1));
}

// The k-th largest of the keys >= lo in buf[0, n) (k <= their number), by an
// 8-bit-digit radix select with a shared histogram: only for a CTA that holds
// more than top_k keys above the bound, which the bound makes rare.
__device__ __noinline__ unsigned long long sq_kth_largest(const uint64_t *buf, int n, uint64_t lo, int k,
                                                          SQHdr *m, int et) {
    unsigned long long prefix = 0ull, pmask = 0ull;
    int remaining = k;
    for (int shift = 56; shift >= 0; shift -= 8) {
        for (int i = et; i < 256; i += kSQEpi) m->hist[i] = 0;
        named_bar(kSQBarTail, kSQEpi);
        for (int j = et; j < n; j += kSQEpi) {
            const uint64_t key = buf[j];
            if (key >= lo && (key & pmask) == prefix) atomicAdd(&m->hist[(key >> shift) & 255u], 1);
        }
        named_bar(kSQBarTail, kSQEpi);
        if (et < 32) {
            int d, above, inbin;
            scan_digit<8>(m->hist, remaining, et, d, above, inbin);
            if (et == 0) {
                m->kth = prefix | (static_cast<unsigned long long>(d) << shift);
                m->ovf_off = remaining - above;
            }
        }
        named_bar(kSQBarTail, kSQEpi);
        prefix = m->kth;
        remaining = m->ovf_off;
        pmask |= 255ull << shift;
        named_bar(kSQBarTail, kSQEpi);
    }
    return prefix;  // keys are unique: exactly one key has all 64 bits equal to it
}

template <int H>
__global__ void __launch_bounds__(kSQThreads, 1)
    stream_select_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_q,
                         const __grid_constant__ ScoreParams p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    const SQLayout L = sq_layout(p.D, H, p.esize, p.kstages, p.cap);
    SQHdr *m = reinterpret_cast<SQHdr *>(smem);
    uint8_t *k_smem = smem + L.k_off;
    uint8_t *q_smem = smem + L.q_off;
    float *w_s = reinterpret_cast<float *>(smem + L.w_off);
    uint64_t *buf = reinterpret_cast<uint64_t *>(smem + L.buf_off);
    uint16_t *mask_s = reinterpret_cast<uint16_t *>(smem + L.mask_off);
    float *ks_s = reinterpret_cast<float *>(smem + L.ks_off);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = blockIdx.x % p.n_groups;
    const int split = blockIdx.x / p.n_groups;
    const long long t = g;  // one query per group
    const int S = p.splits, K = p.top_k;
    const int nchunk = p.D * p.esize / 128;  // 128-byte column chunks of a row
    const int cw = 128 / p.esize;
    const uint32_t tile_bytes = static_cast<uint32_t>(kBM * p.D * p.esize);
    volatile int *abort_flag = &m->abort_flag;

    // Prologue. Nothing before the dependency wait touches global memory: under
    // a programmatic launch it overlaps the previous grid's tail.
    if (threadIdx.x == 0) {
        for (int s = 0; s < p.kstages; ++s) {
            mbar_init(&m->k_full[s], 1);
            mbar_init(&m->k_empty[s], 1);
        }
        for (int a = 0; a < kSQAcc; ++a) {
            mbar_init(&m->acc_full[a], 1);
            mbar_init(&m->acc_empty[a], 4);  // the four warps of the group that consumed it
        }
        mbar_init(&m->q_full, 1);
        mbar_init(&m->mma_done, 1);
        mbar_init(&m->never, 1);
        mbar_init(&m->side_full, 1);
        m->abort_flag = 0;
        m->done_counted = 0;
        m->cnt = 0;
        m->live_bound = 0ull;
        m->bound = 0ull;
        fence_mbar_init();
        tma_prefetch_desc(&tm_k);
        tma_prefetch_desc(&tm_q);
        asm volatile("griddepcontrol.wait;" ::: "memory");
        const int tile0 = split * p.tiles_per_split;
        const int ntl = max(0, min(p.tiles_per_split, p.n_tiles - tile0));
        m->tile0 = tile0;
        m->ntl = ntl;
        // The key-side data first (the mask bits and key scales of the CTA's keys: small,
        // needed by the first tile, and behind the K stream they would wait for most of it),
        // as bulk copies of the 16-byte aligned part; the epilogue loads the rest itself.
        const long long key0 = static_cast<long long>(tile0) * kBM;
        const long long valid = max(0ll, min(static_cast<long long>(ntl) * kBM, p.n_kv - key0));
        const uint32_t mbytes = (p.mask != nullptr && (p.side_bulk & 1)) ? static_cast<uint32_t>(valid * 2) & ~15u : 0u;
        const uint32_t kbytes = (p.k_scale != nullptr && (p.side_bulk & 2)) ? static_cast<uint32_t>(valid * 4) & ~15u : 0u;
        if (mbytes + kbytes > 0u) {
            mbar_arrive_expect_tx(&m->side_full, mbytes + kbytes);
            if (mbytes) bulk_load(mask_s, p.mask + t * p.n_kv + key0, mbytes, &m->side_full);
            if (kbytes) bulk_load(ks_s, p.k_scale + key0, kbytes, &m->side_full);
        } else {
            mbar_arrive(&m->side_full);
        }
        m->m_staged = static_cast<int>(mbytes / 2u);
        m->k_staged = static_cast<int>(kbytes / 4u);
        // q next: the first MMA needs it, and it would otherwise queue behind the K stages
        if (ntl > 0) {
            mbar_arrive_expect_tx(&m->q_full, static_cast<uint32_t>(H * p.D * p.esize));
            for (int c = 0; c < nchunk; ++c)
                tma_load_2d(q_smem + c * H * 128, &tm_q, c * cw, static_cast<int>(t * H), &m->q_full);
        }
        for (int i = 0; i < ntl && i < p.kstages; ++i) {
            mbar_arrive_expect_tx(&m->k_full[i], tile_bytes);
            for (int c = 0; c < nchunk; ++c)
                tma_load_2d(k_smem + i * L.stage + c * kBM * 128, &tm_k, c * cw, (tile0 + i) * kBM, &m->k_full[i]);
        }
    }
    if (warp == 1) {
        tmem_alloc(&m->tmem_base, p.tmem_cols);
        tmem_relinquish();
    }
    asm volatile("griddepcontrol.wait;" ::: "memory");
    if (warp >= 10) {
        const int h = threadIdx.x - 320;
        // 8-bit operands: w relu(q_scale x) = (w q_scale) relu(x) for q_scale >= 0
        if (h < H) w_s[h] = p.w[t * H + h] * (p.q_scale != nullptr ? p.q_scale[t * H + h] : 1.f);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = m->tmem_base;
    const int tile0 = m->tile0;
    const int ntl = m->ntl;

    if (warp == 0) {
        // ---------------------------------------------------------- TMA producer
        if (lane == 0) {
            int issued = ntl < p.kstages ? ntl : p.kstages;
            for (int i = issued; i < ntl; ++i) {
                const int s = i % p.kstages;
                const uint32_t ph = static_cast<uint32_t>(i / p.kstages) & 1u;
                if (!mbar_wait(&m->k_empty[s], ph ^ 1u, abort_flag, 1, p.wait_limit)) break;
                mbar_arrive_expect_tx(&m->k_full[s], tile_bytes);
                for (int c = 0; c < nchunk; ++c)
                    tma_load_2d(k_smem + s * L.stage + c * kBM * 128, &tm_k, c * cw, (tile0 + i) * kBM, &m->k_full[s]);
                issued = i + 1;
            }
            // loads still in flight must land before the CTA may exit
            for (int i = max(0, issued - p.kstages); i < issued; ++i) {
                int dummy = 0;
                mbar_wait(&m->k_full[i % p.kstages], static_cast<uint32_t>(i / p.kstages) & 1u, &dummy, 1,
                          p.wait_limit);
            }
            if (ntl > 0) {
                int dummy = 0;
                mbar_wait(&m->q_full, 0, &dummy, 1, p.wait_limit);
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        // ----------------------------------------------------------- MMA issuer
        if (lane == 0) {
            const uint64_t q_desc = smem_desc_sw128(smem_u32(q_smem)), k_desc = smem_desc_sw128(smem_u32(k_smem));
            bool ok = ntl == 0 || mbar_wait(&m->q_full, 0, abort_flag, 2, p.wait_limit);
            tc_fence_after();
            // four MMAs (one per 32 bytes of a row) per 128-byte column chunk, 1 or 2 chunks
            const bool f8 = p.esize == 1;
            const bool two_chunks = p.D * p.esize == 256;
            const uint64_t step_k = static_cast<uint64_t>(kBM * 128) >> 4, step_q = static_cast<uint64_t>(H * 128) >> 4;
            for (int i = 0; ok && i < ntl; ++i) {
                const int s = i % p.kstages, a = i % kSQAcc;
                if (!mbar_wait(&m->k_full[s], static_cast<uint32_t>(i / p.kstages) & 1u, abort_flag, 2, p.wait_limit))
                    break;
                if (i >= kSQAcc &&
                    !mbar_wait(&m->acc_empty[a], (static_cast<uint32_t>(i / kSQAcc) & 1u) ^ 1u, abort_flag, 2,
                               p.wait_limit))
                    break;
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(a * H);
                const uint64_t ks = k_desc + ((static_cast<uint32_t>(s) * L.stage) >> 4);
                if (f8) {
                    umma_quad<true>(d_tmem, ks, q_desc, p.idesc, 0u);
                } else {
                    umma_quad<false>(d_tmem, ks, q_desc, p.idesc, 0u);
                    if (two_chunks) umma_quad<false>(d_tmem, ks + step_k, q_desc + step_q, p.idesc, 1u);
                }
                umma_commit(&m->k_empty[s]);
                umma_commit(&m->acc_full[a]);
            }
            // every MMA issued has finished before the tensor memory may be freed
            umma_commit(&m->mma_done);
            int dummy = 0;
            mbar_wait(&m->mma_done, 0, &dummy, 2, p.wait_limit);
        }
        __syncwarp();
    } else if (warp < 10) {
        // ------------------------------------------------------ streaming groups
        const int sg = (warp - 2) >> 2;                // group: tiles sg, sg + 2, ...
        const int quarter = warp & 3;                  // TMEM lane quarter of this warp
        const int row = quarter * 32 + lane;           // this thread's key within a tile
        const uint16_t *mrow = p.mask != nullptr ? p.mask + t * p.n_kv : nullptr;
        // keys [tile0 * 128, + m_staged) have their mask bits (k_staged: key scales) in shared memory
        const int m_staged = m->m_staged, k_staged = m->k_staged;
        int dummy = 0;
        const bool side_ok = mbar_wait(&m->side_full, 0, &dummy, 3, p.wait_limit);
        auto mask_bits = [&](int i) -> uint16_t {
            const int j = i * kBM + row;  // the key's place in the CTA
            const long long s = static_cast<long long>(tile0) * kBM + j;
            if (mrow == nullptr || i >= ntl || s >= p.n_kv) return static_cast<uint16_t>(0);
            return (j < m_staged && side_ok) ? mask_s[j] : __ldg(mrow + s);
        };
        unsigned long long umx = 0ull;  // this row's largest key so far (the certificates)
        bool published = false;
        auto publish = [&]() {
            m->comb[sg][row] = umx;
            __syncwarp();
            asm volatile("bar.arrive %0, %1;" ::"r"(kSQBarPub), "r"(kSQEpi) : "memory");
            published = true;
        };
        uint16_t mnext = mask_bits(sg);
        bool ok = true;
        for (int i = sg; i < ntl; i += 2) {
            const int a = i % kSQAcc;
            const long long s = static_cast<long long>(tile0 + i) * kBM + row;
            const bool s_ok = s < p.n_kv;
            const uint16_t mbits = mnext;  // loaded one of this group's tiles ago
            mnext = mask_bits(i + 2);
            // (8-bit operands) relu(k_scale x) = k_scale relu(x): the key scale multiplies the sum
            const int jk = i * kBM + row;
            const float ksc = (p.k_scale == nullptr || !s_ok) ? 1.f : ((jk < k_staged && side_ok) ? ks_s[jk] : __ldg(p.k_scale + s));
            ok = mbar_wait(p.fault == 2 ? &m->never : &m->acc_full[a], static_cast<uint32_t>(i / kSQAcc) & 1u,
                           abort_flag, 3, p.wait_limit);
            ok = __all_sync(0xFFFFFFFFu, ok);  // warp-uniform before the .sync.aligned TMEM loads
            tc_fence_after();
            if (!ok) break;
            // a warp whose 32 keys are all masked skips the sum: the score is -inf whatever it is
            const bool hidden = __all_sync(0xFFFFFFFFu, mbits == kF16NegInf);
            const float hs = hidden ? 0.f
                                    : sq_head_sum<H>(tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) +
                                                         static_cast<uint32_t>(a * H),
                                                     w_s);
            const float score = hidden ? __uint_as_float(0xFF800000u) : fmaf(hs, ksc, f16_bits_to_float(mbits));
            const uint64_t key = s_ok ? make_key(score, static_cast<uint32_t>(s)) : 0ull;
            umx = key > umx ? key : umx;
            // below the certified bound (once the merge group has it) a key cannot reach the output
            const bool keep = key >= *reinterpret_cast<volatile unsigned long long *>(&m->live_bound);
            warp_append(buf, &m->cnt, key, s_ok && keep, lane);
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&m->acc_empty[a]);
            if (!published && i + 2 >= p.f_pub) publish();
        }
        if (!published) publish();
    } else {
        // ------------------------------------------- merge group: the certified bound
        const int mt = threadIdx.x - 320;  // 0..127: a row
        const int mw = mt >> 5;
        asm volatile("bar.sync %0, %1;" ::"r"(kSQBarPub), "r"(kSQEpi) : "memory");
        const unsigned long long v = m->comb[0][mt] > m->comb[1][mt] ? m->comb[0][mt] : m->comb[1][mt];
        // a row without keys gets a small stand-in (1..128, below every real key) so all 128 values differ
        const unsigned long long srt = warp_sort_desc_u64(row_value(v, mt), lane);
        m->srt[mt] = srt;
        if (split == 0 && mt == 0) p.f_count[t] = 0;  // the overflow list (read after the second meeting)
        named_bar(kSQBarM, 128);
        // A. the CTA holds >= r keys >= the r-th largest row maximum: publish r = 1, 2, 4, ..., 128
        int rank = lane;
#pragma unroll
        for (int o = 1; o < 4; ++o) rank += count_above32(m->srt + ((mw + o) & 3) * 32, srt);
        if ((rank & (rank + 1)) == 0)
            // level-major ([row][level][split]): a level's certificates are one contiguous run
            p.f_stats[(t * kFusedLevels + (31 - __clz(rank + 1))) * S + split] = srt > 255ull ? srt : 0ull;
        named_bar(kSQBarM, 128);
        bool ok = true;
        if (mt == 0) ok = sq_grid_wait(p, g, static_cast<unsigned>(S) + (p.fault == 3 ? 1u : 0u), abort_flag);
        named_bar(kSQBarM, 128);
        if (*abort_flag == 0) {
            // B. per level l: at least c = ceil(top_k / 2^l) CTAs hold 2^l keys >= their
            // certificate. The S certificates' scores (ord values) go into 256 bins over their
            // range, by a monotone map (a larger value never lands in a lower bin); the
            // smallest value in the bin holding the c-th largest is <= the c-th largest, so
            // (it << 32) bounds the top_k-th key from below. Warp mw takes levels 2 + mw and
            // 6 + mw, and for a top_k small enough to need them also level mw (levels 0-1);
            // the loads of all of them are in flight together.
            int *hist = m->bhist[mw];
            unsigned *minb = reinterpret_cast<unsigned *>(m->bmin[mw]);
            const unsigned long long *st = reinterpret_cast<const unsigned long long *>(p.f_stats + t * kFusedLevels * S);
            uint32_t o[3][kBoundVPL];
#pragma unroll
            for (int e = 0; e < 3; ++e)
#pragma unroll
                for (int k = 0; k < kBoundVPL; ++k) {
                    const int j = lane + 32 * k, l = e < 2 ? 2 + mw + 4 * e : mw;
                    const bool need = l < kFusedLevels && (e < 2 || mw < 2) && ((K + (1 << l) - 1) >> l) <= S;
                    o[e][k] = (j < S && need) ? static_cast<uint32_t>(__ldcg(st + l * S + j) >> 32) : 0u;
                }
#pragma unroll
            for (int e = 0; e < 3; ++e) {
                const int l = e < 2 ? 2 + mw + 4 * e : mw;
                const int c = (K + (1 << l) - 1) >> l;
                if (l >= kFusedLevels || (e == 2 && mw >= 2) || c > S) continue;  // warp-uniform
                uint32_t lo = ~0u, hi = 0u;
#pragma unroll
                for (int k = 0; k < kBoundVPL; ++k)
                    if (o[e][k] != 0u) {
                        lo = o[e][k] < lo ? o[e][k] : lo;
                        hi = o[e][k] > hi ? o[e][k] : hi;
                    }
                lo = __reduce_min_sync(0xFFFFFFFFu, lo);
                hi = __reduce_max_sync(0xFFFFFFFFu, hi);
                if (lo > hi) continue;  // no certificate at this level (uniform)
                for (int b = lane; b < 256; b += 32) {
                    hist[b] = 0;
                    minb[b] = ~0u;
                }
                __syncwarp();
                const float scale = 256.f / (static_cast<float>(hi - lo) + 1.f);
                int nz = 0;
#pragma unroll
                for (int k = 0; k < kBoundVPL; ++k)
                    if (o[e][k] != 0u) {
                        const int bin = min(255, static_cast<int>(static_cast<float>(o[e][k] - lo) * scale));
                        atomicAdd(&hist[bin], 1);
                        atomicMin(&minb[bin], o[e][k]);
                        ++nz;
                    }
                nz = __reduce_add_sync(0xFFFFFFFFu, nz);
                __syncwarp();
                if (nz >= c) {
                    int d, ab, inb;
                    scan_digit<8>(hist, c, lane, d, ab, inb);
                    if (lane == 0 && d >= 0) atomicMax(&m->bound, static_cast<unsigned long long>(minb[d]) << 32);
                }
                __syncwarp();  // the next level clears the bins
            }
        }
        named_bar(kSQBarM, 128);
        if (mt == 0) m->live_bound = m->bound;
        (void)ok;
    }

    if (warp >= 2) {
        // ------------------------------------------------------------------ tail
        const int et = threadIdx.x - 64;
        asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
        const bool all_ok = !named_bar_or(kSQBarTail, kSQEpi, *abort_flag != 0);
        if (all_ok) {
            const uint64_t B = m->bound > 0ull ? m->bound : 1ull;  // no certificate: every key is a candidate
            const int n = m->cnt;
            int c = 0;
            for (int j = et; j < n; j += kSQEpi) c += buf[j] >= B ? 1 : 0;
            int mine = 0;
            int pos = block_excl_scan<kSQEpi>(c, et, kSQBarTail, m->wtot, &mine);
            uint64_t *reg = p.f_reg + (t * S + split) * kSQRegion;
            for (int j = et; j < n; j += kSQEpi) {
                const uint64_t key = buf[j];
                if (key >= B) {
                    if (pos < kSQRegion - 1) reg[1 + pos] = key;
                    ++pos;
                }
            }
            for (int j = mine + et; j < kSQRegion - 1; j += kSQEpi) reg[1 + j] = 0ull;
            if (et == 0) reg[0] = static_cast<uint64_t>(mine);
            if (mine > kSQRegion - 1) {
                // more keys than the region holds: all of them (at most top_k, this CTA's
                // own top ones) also go to the query's overflow list
                const uint64_t lo = mine > K ? sq_kth_largest(buf, n, B, K, m, et) : B;
                const int take = mine > K ? K : mine;
                if (et == 0) m->ovf_off = atomicAdd(&p.f_count[t], take);
                named_bar(kSQBarTail, kSQEpi);
                int c2 = 0;
                for (int j = et; j < n; j += kSQEpi) c2 += buf[j] >= lo ? 1 : 0;
                int dummy = 0;
                int pos2 = m->ovf_off + block_excl_scan<kSQEpi>(c2, et, kSQBarTail, m->wtot, &dummy);
                uint64_t *dst = p.f_cand + t * p.f_cap;
                for (int j = et; j < n; j += kSQEpi)
                    if (buf[j] >= lo) dst[pos2++] = buf[j];
            }
            // the second meeting: every region (and overflow list) is written
            bool ok = true;
            if (et == 0) {
                ok = sq_grid_wait(p, g, 2u * static_cast<unsigned>(S), abort_flag);
                if (ok) {
                    // every CTA has arrived at both meetings: once all have also seen this one
                    // pass (counted in f_done, after their acquiring poll), the last clears the
                    // counters for the next launch; its latency overlaps the loads below
                    m->done_counted = 1;
                    if (atomicAdd(p.f_done + g, 1u) == static_cast<unsigned>(S) - 1u) {
                        p.f_bar[g] = 0u;
                        p.f_done[g] = 0u;
                    }
                }
            }
            if (!named_bar_or(kSQBarTail, kSQEpi, !ok || *abort_flag != 0)) {
                // Every region, one warp per region at a time (lane i reads slot i; lane 0's slot
                // is the count). A region's keys count unless it overflowed (its keys are then in
                // the overflow list, which comes after them).
                const int n_ovf = __ldcg(&p.f_count[t]);
                const unsigned long long *src =
                    reinterpret_cast<const unsigned long long *>(p.f_reg + t * S * kSQRegion);
                constexpr int EW = kSQEpi / 32;  // epilogue warps
                constexpr int RPW = 13;          // regions a warp holds in registers: S <= 152 < 13 EW
                const int ew = et >> 5;
                unsigned long long rv[RPW];
#pragma unroll
                for (int u = 0; u < RPW; ++u) {
                    const int r = ew + u * EW;
                    rv[u] = r < S ? __ldcg(src + r * kSQRegion + lane) : 0ull;
                }
                unsigned kb[RPW];  // per region: which lanes hold a key that counts
                int wcount = 0;
#pragma unroll
                for (int u = 0; u < RPW; ++u) {
                    const unsigned long long h = __shfl_sync(0xFFFFFFFFu, rv[u], 0);
                    const bool key = lane != 0 && rv[u] > 0xFFFFFFFFull && h <= kSQRegion - 1;
                    kb[u] = __ballot_sync(0xFFFFFFFFu, key);
                    wcount += __popc(kb[u]);
                }
                if (lane == 0) m->wtot[ew] = wcount;
                named_bar(kSQBarTail, kSQEpi);
                int base = 0, n_reg = 0;
#pragma unroll
                for (int w = 0; w < EW; ++w) {
                    const int x = m->wtot[w];
                    base += w < ew ? x : 0;
                    n_reg += x;
                }
                unsigned long long *cand = reinterpret_cast<unsigned long long *>(k_smem);  // the idle K stages
#pragma unroll
                for (int u = 0; u < RPW; ++u) {
                    if ((kb[u] >> lane) & 1u) cand[base + __popc(kb[u] & ((1u << lane) - 1u))] = rv[u];
                    base += __popc(kb[u]);
                }
                // (the overflow list, if any, stays in global memory: it can exceed shared memory)
                const unsigned long long *ovf = reinterpret_cast<const unsigned long long *>(p.f_cand + t * p.f_cap);
                named_bar(kSQBarTail, kSQEpi);
                const int total = n_reg + n_ovf;
                // rank this CTA's slice: keys are unique, so a key's rank is the number of larger ones
                const int per = (total + S - 1) / S;
                const int lo = split * per, hi = min(total, lo + per);
                for (int ci = lo + ew; ci < hi; ci += kSQEpi / 32) {
                    const unsigned long long x = ci < n_reg ? cand[ci] : __ldcg(ovf + (ci - n_reg));
                    int r = 0, r1 = 0;
                    int y = lane;
                    for (; y + 32 < n_reg; y += 64) {
                        r += cand[y] > x ? 1 : 0;
                        r1 += cand[y + 32] > x ? 1 : 0;
                    }
                    if (y < n_reg) r += cand[y] > x ? 1 : 0;
                    for (int z = lane; z < n_ovf; z += 32) r += __ldcg(ovf + z) > x ? 1 : 0;
                    r = __reduce_add_sync(0xFFFFFFFFu, r + r1);
                    if (lane == 0 && r < K) {
                        int32_t idx;
                        float sc;
                        decode_key(x, idx, sc);
                        p.out_idx[t * K + r] = idx;
                        p.out_score[t * K + r] = sc;
                    }
                }
                if (split == 0)  // fewer candidates than top_k only without a certified bound
                    for (int j = total + et; j < K; j += kSQEpi) {
                        p.out_idx[t * K + j] = -1;
                        p.out_score[t * K + j] = __uint_as_float(0xFF800000u);
                    }
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (threadIdx.x == 0 && m->done_counted == 0) {
        // a CTA that did not pass the second meeting (a wait ran out) counts itself here;
        // every CTA gets here (all waits are bounded), so the group's last one clears the
        // counters for the next launch
        __threadfence();
        if (atomicAdd(p.f_done + g, 1u) == static_cast<unsigned>(S) - 1u) {
            p.f_bar[g] = 0u;
            p.f_done[g] = 0u;
        }
    }
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, p.tmem_cols);
    }
}

}  // namespace lid
