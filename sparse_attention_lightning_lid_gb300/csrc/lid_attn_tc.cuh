// lid_attn_tc.cuh -- sparse attention over the selected latent rows on the
// 5th-generation tensor cores (tcgen05), for 64 query heads per CTA.
//
// Same operation as lid_attn.cuh ("Eval bug: DeepSeek-V4-Flash
// lightning-indexer ..." (llama.cpp issue 25468), root-cause comment;
// "deepseek v4 support" (llama.cpp PR 22378), batched-prefill commit:
// Q*K^T -> softmax -> *V over the 512-wide MLA latent rows). One CTA takes one
// query row, 64 heads and one range of selections, in chunks of 128 keys:
//
//   producer warps (0-3): gather the chunk's 128 rows by index with 16-byte
//                   cp.async into 8 regions of 128 rows x 64 dims (the
//                   128-byte swizzle: piece p of row r at p ^ (r & 7)), region
//                   b holding dims 64b..64b+63; each region is handed to the
//                   tensor core (proxy fence, mbarrier) as soon as it lands.
//                   (TMA's four-row gather moves 512 bytes per copy and its
//                   per-copy cost made it several times slower here.)
//   MMA thread (warp 12): S^T = K . Q^T into tensor memory (M = 128 keys,
//                   N = 64 heads, K = 512: the regions as K-major A, Q as
//                   K-major B), then O^T += V^T . P^T (M = 128 dims per block,
//                   N = 64 heads, K = 128 keys: the same regions read as an
//                   MN-major A, P^T as an MN-major B);
//   softmax warps (4-11): thread (k, half) owns key row k of S^T (tensor-
//                   memory lane k) for heads 32*half..32*half+31: per-head
//                   chunk maxima through a halving butterfly and shared
//                   memory, a running maximum per head that moves only when a
//                   chunk exceeds it by more than 2^8 (weights stay below 2^8
//                   and the output accumulator is rescaled only then),
//                   p = 2^(s*scale*log2e - m) summed in fp32 per thread and
//                   stored as 16-bit floats into P^T (row k); at the end they
//                   normalise O^T into shared memory, which one bulk copy
//                   writes out.
//
// Tensor memory: S^T in two 64-column buffers, O^T in four blocks of 64
// columns (dims 0..127, 128..255, ...), 384 of the 512 columns allocated.
// Keys and values are the same staged rows, so each selected row crosses the
// chip once per CTA.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "lid_attn.cuh"
#include "lid_ptx.cuh"

namespace lid {
namespace attn {

constexpr int kTcKeys = 128;                 // keys per chunk (M of S^T)
constexpr int kTcHeads = 64;                 // heads per CTA (N)
constexpr int kTcRegions = 8;                // 64-dim regions of a chunk
constexpr int kTcRegionBytes = kTcKeys * 128;
constexpr int kTcThreads = 416;              // warps 0-3 producers, 4-11 softmax, 12 MMA (128 registers:
                                             // an SM sub-partition holds 4 of the 13 warps)
constexpr int kTcMmaWarp = 12;
constexpr float kTcTau = 8.0f;               // log2 slack before the running maximum moves

struct TcSmem {
    static constexpr int kQ = 0;                                      // 8 x (64 heads x 128 B)
    static constexpr int kRing = kQ + kTcRegions * kTcHeads * 128;    // 8 x (128 keys x 128 B)
    static constexpr int kP = kRing + kTcRegions * kTcRegionBytes;    // P^T: 128 keys x 128 B
    static constexpr int kBar = kP + kTcKeys * 128;
    static constexpr int kNumBars = 1 + kTcRegions + kTcRegions / 2 + 2 + 2 + 3;
    static constexpr int kRed = kBar + 256;                           // [4][64] floats
    static constexpr int kMRun = kRed + 4 * 64 * 4;
    static constexpr int kMUse = kMRun + 64 * 4;
    static constexpr int kAlpha = kMUse + 64 * 4;
    static constexpr int kMisc = kAlpha + 64 * 4;                     // flags, tmem base, abort
    static constexpr int kEnd = kMisc + 64;
    static constexpr int kTotal = kEnd + 1024;                        // slack to align the base to 1024
};

struct TcBars {
    uint64_t q_full;
    uint64_t region_full[kTcRegions];
    uint64_t region_empty[kTcRegions / 2];  // per pair of regions (one block of 128 dims of V)
    uint64_t s_full[2];
    uint64_t s_empty[2];
    uint64_t p_full, p_empty, o_full;
};
static_assert(sizeof(TcBars) == TcSmem::kNumBars * 8 && sizeof(TcBars) <= 256, "barrier area");

struct TcMisc {
    int rescale[2];
    uint32_t tmem_base;
    int abort_flag;
};

__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t *r) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(
            taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
        "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
        : "memory");
}

__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Matrix descriptor with explicit offsets (128-byte swizzle). For an MN-major
// operand, `lbo` is the distance between 64-element atoms along M (or N) and
// `sbo` the distance between groups of 8 rows along K.
__device__ __forceinline__ uint64_t desc_sw128(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
    return static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4) | (static_cast<uint64_t>(lbo >> 4) << 16) |
           (static_cast<uint64_t>(sbo >> 4) << 32) | (static_cast<uint64_t>(1) << 46) |
           (static_cast<uint64_t>(2) << 61);
}

// Halving butterfly over the 32 lanes of a warp: v[0..31] in, and lane l ends
// with the reduction over the warp of value l in v[0].
template <bool MAX>
__device__ __forceinline__ void warp_halving32(float (&v)[32], int lane) {
#pragma unroll
    for (int half = 16, bit = 16; half >= 1; half >>= 1, bit >>= 1) {
        const bool up = (lane & bit) != 0;
#pragma unroll
        for (int j = 0; j < half; ++j) {
            const float keep = up ? v[half + j] : v[j];
            const float send = up ? v[j] : v[half + j];
            const float got = __shfl_xor_sync(0xffffffffu, send, bit);
            v[j] = MAX ? fmaxf(keep, got) : keep + got;
        }
    }
}

template <int R>
__device__ __forceinline__ void cp_async_wait_n() {
    asm volatile("cp.async.wait_group %0;" ::"n"(R) : "memory");
}

// Hand region r of the chunk to the tensor core once this thread's copies into
// it have landed (the last 7 - r regions' copies may still be in flight).
template <int R>
__device__ __forceinline__ void region_landed(uint64_t *full) {
    cp_async_wait_n<7 - R>();
    fence_proxy_async_smem();
    mbar_arrive(&full[R]);
}

template <bool F16>
__global__ void __launch_bounds__(kTcThreads, 1)
    sparse_attn_tc_kernel(const __grid_constant__ Params p, long long wait_limit) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    TcBars *bars = reinterpret_cast<TcBars *>(smem + TcSmem::kBar);
    float *red = reinterpret_cast<float *>(smem + TcSmem::kRed);
    float *m_run = reinterpret_cast<float *>(smem + TcSmem::kMRun);
    float *m_use = reinterpret_cast<float *>(smem + TcSmem::kMUse);
    float *alpha_s = reinterpret_cast<float *>(smem + TcSmem::kAlpha);
    TcMisc *misc = reinterpret_cast<TcMisc *>(smem + TcSmem::kMisc);
    volatile int *abort_flag = &misc->abort_flag;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const long long b = blockIdx.x;
    const int split = static_cast<int>(b % p.splits);
    const int hb = static_cast<int>((b / p.splits) % p.head_blocks);
    const long long t = b / (static_cast<long long>(p.splits) * p.head_blocks);
    const int head0 = hb * kTcHeads;
    const int j_lo = split * p.keys_per_split;
    const int j_hi = min(p.top_k, j_lo + p.keys_per_split);
    const int nch = j_hi > j_lo ? (j_hi - j_lo + kTcKeys - 1) / kTcKeys : 0;
    const int32_t *ix = p.idx + t * p.top_k;
    const float *sc = p.sel_score ? p.sel_score + t * p.top_k : nullptr;

    if (threadIdx.x == 0) {
        mbar_init(&bars->q_full, 128);
        for (int i = 0; i < kTcRegions; ++i) mbar_init(&bars->region_full[i], 128);
        for (int i = 0; i < kTcRegions / 2; ++i) mbar_init(&bars->region_empty[i], 1);
        for (int i = 0; i < 2; ++i) {
            mbar_init(&bars->s_full[i], 1);
            mbar_init(&bars->s_empty[i], 256);
        }
        mbar_init(&bars->p_full, 256);
        mbar_init(&bars->p_empty, 1);
        mbar_init(&bars->o_full, 1);
        misc->rescale[0] = misc->rescale[1] = 0;
        misc->abort_flag = 0;
        fence_mbar_init();
    }
    if (threadIdx.x < 64) m_run[threadIdx.x] = -INFINITY;
    if (warp == kTcMmaWarp) {
        tmem_alloc(&misc->tmem_base, 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = misc->tmem_base;
    // nothing global is read before the work this launch depends on is done
    asm volatile("griddepcontrol.wait;" ::: "memory");

    if (warp < 4) {
        // ------------------------------------------------------ gather producers
        const int tid = threadIdx.x;  // 0..127
        {
            const uint16_t *qsrc = p.qa + (t * p.Ha + head0) * kDc;
            const uint32_t q_s = smem_u32(smem + TcSmem::kQ);
            for (int i = tid; i < kTcHeads * 64; i += 128) {
                const int row = i >> 6, piece = i & 63;  // head row, 16-byte piece of its 1 KiB
                const int reg = piece >> 3, ch = piece & 7;
                cp_async16(q_s + reg * kTcHeads * 128 + row * 128 + ((ch ^ (row & 7)) << 4),
                           qsrc + row * kDc + piece * 8);
            }
            asm volatile("cp.async.wait_all;" ::: "memory");
            fence_proxy_async_smem();
            mbar_arrive(&bars->q_full);
        }
        const uint32_t ring_s = smem_u32(smem + TcSmem::kRing);
        const int piece = tid & 7;
        for (int c = 0; c < nch; ++c) {
            // this thread's 8 rows of the chunk: (tid >> 3) + 16 i; a dropped
            // selection reads row 0 (its weight is 0)
            int srow[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const int j = j_lo + c * kTcKeys + (tid >> 3) + 16 * i;
                long long s = -1;
                if (j < j_hi) {
                    s = ix[j];
                    if (sc && sc[j] == -INFINITY) s = -1;
                }
                srow[i] = (s < 0 || s >= p.n_kv) ? 0 : static_cast<int>(s);
            }
            const uint16_t *kv_p = p.kv + piece * 8;
            bool ok = true;
#pragma unroll
            for (int r = 0; r < kTcRegions; ++r) {
                if (c > 0 && ok && (r & 1) == 0 &&
                    !mbar_wait(&bars->region_empty[r >> 1], (c - 1) & 1, abort_flag, 4, wait_limit))
                    ok = false;
                if (ok) {
                    const uint32_t dst = ring_s + r * kTcRegionBytes;
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        const int row = (tid >> 3) + 16 * i;
                        cp_async16(dst + row * 128 + ((piece ^ (row & 7)) << 4),
                                   kv_p + static_cast<long long>(srow[i]) * kDc + 64 * r);
                    }
                }
                cp_async_commit();
            }
            // hand each region over as it lands (also on an abort: nothing is left in flight)
            region_landed<0>(bars->region_full);
            region_landed<1>(bars->region_full);
            region_landed<2>(bars->region_full);
            region_landed<3>(bars->region_full);
            region_landed<4>(bars->region_full);
            region_landed<5>(bars->region_full);
            region_landed<6>(bars->region_full);
            region_landed<7>(bars->region_full);
            if (!ok) break;
        }
    } else if (warp == kTcMmaWarp) {
        // ------------------------------------------------------- MMA issuer
        if (lane == 0) {
            const uint32_t fmt = F16 ? 0u : 1u;
            const uint32_t idesc_s = make_idesc(kTcKeys, kTcHeads, static_cast<int>(fmt));
            const uint32_t idesc_pv = make_idesc(128, kTcHeads, static_cast<int>(fmt)) | (1u << 15) | (1u << 16);
            const uint32_t q_s = smem_u32(smem + TcSmem::kQ);
            const uint32_t ring_s = smem_u32(smem + TcSmem::kRing);
            const uint32_t p_s = smem_u32(smem + TcSmem::kP);
            const uint64_t pdesc = desc_sw128(p_s, kTcRegionBytes, 1024);
            bool ok = nch == 0 || mbar_wait(&bars->q_full, 0, abort_flag, 5, wait_limit);
            tc_fence_after();
            for (int c = 0; ok && c < nch; ++c) {
                const int sb = c & 1;
                if (c >= 2 && !mbar_wait(&bars->s_empty[sb], ((c - 2) >> 1) & 1, abort_flag, 5, wait_limit)) break;
                const uint32_t d_s = tmem + static_cast<uint32_t>(sb * kTcHeads);
                for (int r = 0; ok && r < kTcRegions; ++r) {
                    if (!mbar_wait(&bars->region_full[r], c & 1, abort_flag, 5, wait_limit)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    // four MMAs of 16 dims (32 bytes of the 128-byte rows) each, from one asm block:
                    // the issuing warp shares its scheduler with busy warps
                    umma_quad<false, 2>(d_s, desc_sw128(ring_s + r * kTcRegionBytes, 16, 1024),
                                        desc_sw128(q_s + r * kTcHeads * 128, 16, 1024), idesc_s, r > 0 ? 1u : 0u);
                }
                if (!ok) break;
                umma_commit(&bars->s_full[sb]);
                if (!mbar_wait(&bars->p_full, c & 1, abort_flag, 5, wait_limit)) break;
                tc_fence_after();
#pragma unroll 1
                for (int mb = 0; mb < 4; ++mb) {
                    const uint32_t d_o = tmem + static_cast<uint32_t>(2 * kTcHeads + mb * kTcHeads);
                    // V^T block: dims 128mb.. (regions 2mb, 2mb+1: atoms along M 16 KiB apart), keys along K
                    const uint64_t vd = desc_sw128(ring_s + 2 * mb * kTcRegionBytes, kTcRegionBytes, 1024);
                    // 16 keys = 16 rows of 128 bytes (2048 bytes: 128 descriptor units) per MMA
                    umma_quad<false, 128>(d_o, vd, pdesc, idesc_pv, c > 0 ? 1u : 0u);
                    umma_quad<false, 128>(d_o, vd + 4 * 128, pdesc + 4 * 128, idesc_pv, 1u);
                    umma_commit(&bars->region_empty[mb]);  // regions 2mb, 2mb+1 are free
                }
                umma_commit(&bars->p_empty);
            }
            // every MMA issued so far has finished before the results are read or
            // the tensor memory is freed
            umma_commit(&bars->o_full);
            int dummy = 0;
            mbar_wait(&bars->o_full, 0, &dummy, 5, wait_limit);
        }
        __syncwarp();
    } else {
        // ---------------------------------------------------- softmax, output
        const int sw = warp - 4;             // 0..7
        const int quarter = sw & 3;          // tensor-memory lane quarter (= warp % 4)
        const int half = sw >> 2;            // heads 32*half .. 32*half + 31
        const int k = quarter * 32 + lane;   // key row of a chunk = tensor-memory lane
        const int ts = sw * 32 + lane;       // 0..255
        const uint32_t lane_base = static_cast<uint32_t>(quarter * 32) << 16;
        const uint32_t p_row = smem_u32(smem + TcSmem::kP) + k * 128;
        float l_acc[32];
#pragma unroll
        for (int h = 0; h < 32; ++h) l_acc[h] = 0.f;
        bool ok = true;
        for (int c = 0; c < nch; ++c) {
            const int j = j_lo + c * kTcKeys + k;
            bool valid = false;
            if (j < j_hi) {
                const long long s = ix[j];
                valid = s >= 0 && s < p.n_kv && !(sc && sc[j] == -INFINITY);
            }
            const int sb = c & 1;
            // (a failed wait is voted on at the next group barrier, so the group leaves together)
            if (!mbar_wait(&bars->s_full[sb], (c >> 1) & 1, abort_flag, 6, wait_limit)) ok = false;
            tc_fence_after();
            const uint32_t t_s = tmem + lane_base + static_cast<uint32_t>(sb * kTcHeads + half * 32);
            float v[32];
            tmem_ld32(t_s, reinterpret_cast<uint32_t *>(v));
            tmem_wait_ld();
#pragma unroll
            for (int h = 0; h < 32; ++h) v[h] = valid ? v[h] * p.scale_log2 : -INFINITY;
            warp_halving32<true>(v, lane);  // lane l: head 32*half + l over the warp's 32 keys
            red[quarter * 64 + half * 32 + lane] = v[0];
            if (named_bar_or(1, 256, !ok || *abort_flag != 0)) {
                ok = false;
                break;
            }
            if (ts < 64) {
                const float mc = fmaxf(fmaxf(red[ts], red[64 + ts]), fmaxf(red[128 + ts], red[192 + ts]));
                const float mo = m_run[ts];
                float mn = mo, al = 1.f;
                if (mc > mo + kTcTau) {  // also when nothing was valid before (mo = -inf)
                    mn = mc;
                    al = exp2f(mo - mn);
                    if (c > 0 && mo != -INFINITY) misc->rescale[sb] = 1;
                }
                m_run[ts] = mn;
                m_use[ts] = mn == -INFINITY ? 0.f : mn;
                alpha_s[ts] = al;
            }
            named_bar(1, 256);
            if (ts == 0) misc->rescale[sb ^ 1] = 0;  // every thread read it a chunk ago
            const bool resc = misc->rescale[sb] != 0;
            // the weights of this key for the half's 32 heads
            tmem_ld32(t_s, reinterpret_cast<uint32_t *>(v));
            tmem_wait_ld();
            tc_fence_before();
            mbar_arrive(&bars->s_empty[sb]);
            const float4 *mu4 = reinterpret_cast<const float4 *>(m_use + half * 32);
#pragma unroll
            for (int h4 = 0; h4 < 8; ++h4) {
                const float4 mu = mu4[h4];
                v[4 * h4 + 0] = valid ? exp2f(v[4 * h4 + 0] * p.scale_log2 - mu.x) : 0.f;
                v[4 * h4 + 1] = valid ? exp2f(v[4 * h4 + 1] * p.scale_log2 - mu.y) : 0.f;
                v[4 * h4 + 2] = valid ? exp2f(v[4 * h4 + 2] * p.scale_log2 - mu.z) : 0.f;
                v[4 * h4 + 3] = valid ? exp2f(v[4 * h4 + 3] * p.scale_log2 - mu.w) : 0.f;
            }
            const float *al_h = alpha_s + half * 32;
            if (resc) {
#pragma unroll
                for (int h = 0; h < 32; ++h) l_acc[h] *= al_h[h];
            }
#pragma unroll
            for (int h = 0; h < 32; ++h) l_acc[h] += v[h];
            // P^T and O^T are free once the previous chunk's products are done (already so
            // when S of this chunk is: the tensor core runs the products in issue order)
            if (c > 0 && !mbar_wait(&bars->p_empty, (c - 1) & 1, abort_flag, 6, wait_limit)) ok = false;
            tc_fence_after();
#pragma unroll
            for (int q = 0; q < 4; ++q) {  // 8 heads (16 bytes) per store, swizzled by row
                const uint32_t w0 = pack2<F16>(v[8 * q + 0], v[8 * q + 1]);
                const uint32_t w1 = pack2<F16>(v[8 * q + 2], v[8 * q + 3]);
                const uint32_t w2 = pack2<F16>(v[8 * q + 4], v[8 * q + 5]);
                const uint32_t w3 = pack2<F16>(v[8 * q + 6], v[8 * q + 7]);
                asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(p_row + (((half * 4 + q) ^ (k & 7)) << 4)),
                             "r"(w0), "r"(w1), "r"(w2), "r"(w3)
                             : "memory");
            }
            if (resc) {
                // rare: the running maximum of some head moved; rescale the output
                // columns of those heads (the products of the previous chunks are done)
#pragma unroll 1
                for (int piece = 0; piece < 8; ++piece) {  // 4 blocks x 2 pieces of 16 heads
                    const int mb = piece >> 1, h0 = (piece & 1) * 16;
                    const uint32_t t_o =
                        tmem + lane_base + static_cast<uint32_t>(2 * kTcHeads + mb * kTcHeads + half * 32 + h0);
                    uint32_t o[16];
                    tmem_ld16(t_o, o);
                    tmem_wait_ld();
#pragma unroll
                    for (int h = 0; h < 16; ++h) o[h] = __float_as_uint(__uint_as_float(o[h]) * al_h[h0 + h]);
                    tmem_st16(t_o, o);
                }
                tmem_wait_st();
            }
            fence_proxy_async_smem();
            tc_fence_before();
            mbar_arrive(&bars->p_full);
        }
        // ---- the sums per head, then the normalised output
        if (ok && nch > 0 && !mbar_wait(&bars->o_full, 0, abort_flag, 6, wait_limit)) ok = false;
        const bool all_ok = !named_bar_or(1, 256, !ok || *abort_flag != 0);
        warp_halving32<false>(l_acc, lane);  // lane l: head 32*half + l summed over the warp's keys
        red[quarter * 64 + half * 32 + lane] = l_acc[0];
        named_bar(1, 256);
        float *lsum = alpha_s;
        float *inv_s = m_use;  // the multiplier of each head's row: 1 / l (0 if empty), or 1 for a split's raw rows
        const bool norm = p.splits == 1;
        if (ts < 64) {
            const float l = red[ts] + red[64 + ts] + red[128 + ts] + red[192 + ts];  // l per head
            lsum[ts] = l;
            inv_s[ts] = norm ? (l > 0.f ? 1.f / l : 0.f) : 1.f;
        }
        named_bar(1, 256);
        if (all_ok) {
            tc_fence_after();
            // normalised (or, for a split, raw) rows of the 64 heads, staged [head][512] in the
            // now idle ring and written with one bulk copy
            float *stage = reinterpret_cast<float *>(smem + TcSmem::kRing);
            const float *inv = inv_s + half * 32;
            for (int mb = 0; mb < 4; ++mb) {
                float o[32];
                if (nch > 0) {
                    const uint32_t t_o =
                        tmem + lane_base + static_cast<uint32_t>(2 * kTcHeads + mb * kTcHeads + half * 32);
                    tmem_ld32(t_o, reinterpret_cast<uint32_t *>(o));
                    tmem_wait_ld();
                } else {
#pragma unroll
                    for (int h = 0; h < 32; ++h) o[h] = 0.f;
                }
                const int dim = mb * 128 + k;
#pragma unroll
                for (int h = 0; h < 32; ++h) stage[(half * 32 + h) * kDc + dim] = o[h] * inv[h];
            }
            fence_proxy_async_smem();
            named_bar(1, 256);
            if (ts == 0) {
                float *dst = norm ? p.out + (t * p.Ha + head0) * kDc
                                  : p.part_o + ((t * p.splits + split) * p.Ha + head0) * kDc;
                asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(dst),
                             "r"(smem_u32(stage)), "r"(kTcHeads * kDc * 4)
                             : "memory");
                asm volatile("cp.async.bulk.commit_group;" ::: "memory");
            }
            if (ts < 64) {
                const float l = lsum[ts];
                const float m = m_run[ts];
                if (norm) {
                    p.lse[t * p.Ha + head0 + ts] = l > 0.f ? (m + log2f(l)) * kLn2 : -INFINITY;
                } else {
                    const long long row = (t * p.splits + split) * p.Ha + head0 + ts;
                    *reinterpret_cast<float2 *>(p.part_ml + row * 2) = make_float2(l > 0.f ? m : -INFINITY, l);
                }
            }
            if (ts == 0) asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == kTcMmaWarp) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

}  // namespace attn
}  // namespace lid
