// lid_attn.cuh -- sparse attention over the selected latent rows: the consumer
// of the lightning indexer's top-k.
//
// What it computes ("Eval bug: DeepSeek-V4-Flash lightning-indexer ..."
// (llama.cpp issue 25468), root-cause comment: the top-512 selection feeds the
// CSA layers' attention; "deepseek v4 support" (llama.cpp PR 22378), batched
// prefill commit: Q*K^T -> softmax -> *V over the MLA latent KV, where slots
// masked to -inf contribute nothing): for query row t and head h, over the
// selections J = { j : 0 <= idx[t,j] < n_kv, sel_score[t,j] != -inf },
//   s_j = qa[t,h,:] . kv[idx[t,j],:]
//   out[t,h,:] = sum_j softmax_j(scale * s_j) kv[idx[t,j],:],  lse = log sum_j exp(scale * s_j)
// Keys and values are the same latent rows (Dc = 512 wide).
//
// Layout of the work. A CTA takes one query row, G groups of 16 heads and one
// range of selections (a split), and walks that range in chunks of 64 keys.
// Each chunk's rows are gathered by index from global memory with 16-byte
// cp.async into a two-stage ring (row-major, 1 KiB per row, the 16-byte
// pieces XOR-swizzled by row so that ldmatrix of 8 rows hits 8 distinct bank
// groups). Warp (g, c) of the CTA's 4G warps:
//   S  : 16 heads of group g x keys 16c..16c+15 of the chunk, over all 512
//        dims (mma.sync m16n8k16, fp32 accumulate);
//   softmax: running maximum per head shared by the group's 4 warps through
//        shared memory, p = 2^(s*scale*log2e - m) in fp32, summed in fp32 and
//        rounded to 16 bits into the group's P tile (16 heads x 64 keys);
//   O  : 16 heads x dims 128c..128c+127 += P (16 x 64) . V (64 x 128), V read
//        with ldmatrix.trans from the same staged rows.
// The selections of one query are distinct rows with no reuse across queries,
// so there is no larger shared operand to stage: the contraction per chunk is
// 64 heads x 64 keys x 512 dims twice, which the warp-level MMA covers with
// every staged byte read from shared memory exactly once per consumer warp.
// With one split the CTA normalises and writes out/lse; with several, each
// writes its unnormalised partial (O, running max, sum) and attn_combine
// merges them.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace lid {
namespace attn {

constexpr int kDc = 512;                          // latent row width (elements)
constexpr int kRowBytes = kDc * 2;                // one staged row
constexpr int kChunk = 64;                        // keys per chunk
constexpr int kStageBytes = kChunk * kRowBytes;   // 64 KiB
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

struct Params {
    const uint16_t *qa;       // [n_q][Ha][512]
    const uint16_t *kv;       // [n_kv][512]
    const int32_t *idx;       // [n_q][top_k]
    const float *sel_score;   // [n_q][top_k] or nullptr
    float *out;               // [n_q][Ha][512]           (splits == 1)
    float *lse;               // [n_q][Ha]                (splits == 1)
    float *part_o;            // [n_q][splits][Ha][512]   (splits > 1)
    float *part_ml;           // [n_q][splits][Ha][2]     (running max in log2 units, sum)
    long long n_q, n_kv;
    int Ha, top_k;
    int splits, keys_per_split;  // keys_per_split: a multiple of kChunk
    int head_blocks;             // Ha / (16 G)
    float scale_log2;            // scale * log2(e)
};

template <int G>
struct Smem {
    static constexpr int kQBytes = G * 16 * kRowBytes;
    static constexpr int kPBytes = G * 16 * kChunk * 2;
    static constexpr int kQ = 0;
    static constexpr int kStage = kQ + kQBytes;
    static constexpr int kP = kStage + 2 * kStageBytes;
    static constexpr int kRed = kP + kPBytes;                 // [G][4][16] floats
    static constexpr int kValid = kRed + G * 4 * 16 * 4;      // [2][64] bytes
    static constexpr int kTotal = kValid + 2 * kChunk;
};

__device__ __forceinline__ uint32_t s_u32(const void *p) { return static_cast<uint32_t>(__cvta_generic_to_shared(p)); }

__device__ __forceinline__ void cp_async16(uint32_t dst, const void *src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait1() { asm volatile("cp.async.wait_group 1;" ::: "memory"); }

__device__ __forceinline__ void st_zero16(uint32_t dst) {
    asm volatile("st.shared.v4.u32 [%0], {%1, %1, %1, %1};" ::"r"(dst), "r"(0u) : "memory");
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t (&r)[4]) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t (&r)[4]) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr));
}

// D += A (16x16, row) . B (16x8, col), fp32 accumulate.
template <bool F16>
__device__ __forceinline__ void mma16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    if constexpr (F16) {
        asm volatile(
            "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
            "{%0, %1, %2, %3};"
            : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
            : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
    } else {
        asm volatile(
            "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
            "{%0, %1, %2, %3};"
            : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
            : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
    }
}

// Two fp32 values rounded to nearest into a packed pair of 16-bit floats (lo, hi).
template <bool F16>
__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
    uint32_t r;
    if constexpr (F16) {
        asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    } else {
        asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    }
    return r;
}

// Byte offset of 16-byte piece `piece` of staged row `row` (1 KiB rows).
__device__ __forceinline__ uint32_t row_piece(int row, int piece) {
    return static_cast<uint32_t>(row * kRowBytes + ((piece ^ (row & 7)) << 4));
}

__device__ __forceinline__ void group_bar(int g, int threads) {
    asm volatile("bar.sync %0, %1;" ::"r"(1 + g), "r"(threads) : "memory");
}

// Gather the chunk's rows: selection j in [j0, j0 + 64) of the query's list,
// rows past `j_end`, with an index outside [0, n_kv), or with a -inf
// selection score are zero rows and flagged invalid.
template <int NT>
__device__ __forceinline__ void gather_chunk(const Params &p, long long t, int j0, int j_end, uint32_t stage,
                                             uint8_t *valid) {
    const int tid = threadIdx.x;
    const int32_t *ix = p.idx + t * p.top_k;
    const float *sc = p.sel_score ? p.sel_score + t * p.top_k : nullptr;
#pragma unroll 1
    for (int r = tid >> 3; r < kChunk; r += NT >> 3) {
        const int j = j0 + r;
        bool ok = j < j_end;
        long long s = 0;
        if (ok) {
            s = ix[j];
            ok = s >= 0 && s < p.n_kv && !(sc && sc[j] == -INFINITY);
        }
        if (ok) {
            const uint16_t *src = p.kv + s * kDc;
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const int piece = (tid & 7) + 8 * i;
                cp_async16(stage + row_piece(r, piece), src + piece * 8);
            }
        } else {
#pragma unroll
            for (int i = 0; i < 8; ++i) st_zero16(stage + row_piece(r, (tid & 7) + 8 * i));
        }
        if ((tid & 7) == 0) valid[r] = ok ? 1 : 0;
    }
}

// One CTA: query row t, head groups [G*hb, G*hb + G), selections of split `split`.
template <int G, bool F16>
__global__ void __launch_bounds__(128 * G, 1) sparse_attn_kernel(const __grid_constant__ Params p) {
    constexpr int NT = 128 * G;
    using L = Smem<G>;
    extern __shared__ __align__(1024) uint8_t smem[];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = warp >> 2, c = warp & 3;  // head group of the CTA, key quarter / dim quarter
    const long long b = blockIdx.x;
    const int split = static_cast<int>(b % p.splits);
    const int hb = static_cast<int>((b / p.splits) % p.head_blocks);
    const long long t = b / (static_cast<long long>(p.splits) * p.head_blocks);
    const int head0 = hb * G * 16;

    const uint32_t q_s = s_u32(smem + L::kQ);
    const uint32_t st_s = s_u32(smem + L::kStage);
    const uint32_t p_s = s_u32(smem + L::kP);
    float *red = reinterpret_cast<float *>(smem + L::kRed);
    uint8_t *valid = smem + L::kValid;

    const int j_lo = split * p.keys_per_split;
    const int j_hi = min(p.top_k, j_lo + p.keys_per_split);
    const int nch = j_hi > j_lo ? (j_hi - j_lo + kChunk - 1) / kChunk : 0;

    // nothing global is read before the work this launch depends on is done
    // (a no-op unless launched as a programmatic dependent)
    asm volatile("griddepcontrol.wait;" ::: "memory");
    // queries of the CTA's heads, then the first two chunks
    {
        const uint16_t *qsrc = p.qa + (t * p.Ha + head0) * kDc;
#pragma unroll 1
        for (int i = threadIdx.x; i < G * 16 * 64; i += NT) {
            const int row = i >> 6, piece = i & 63;
            cp_async16(q_s + row_piece(row, piece), qsrc + row * kDc + piece * 8);
        }
    }
    if (nch > 0) gather_chunk<NT>(p, t, j_lo, j_hi, st_s, valid);
    cp_async_commit();
    if (nch > 1) gather_chunk<NT>(p, t, j_lo + kChunk, j_hi, st_s + kStageBytes, valid + kChunk);
    cp_async_commit();

    float o[16][4];
#pragma unroll
    for (int i = 0; i < 16; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
    float m_run[2] = {-INFINITY, -INFINITY};  // running maximum (log2 units) of rows lane/4, lane/4 + 8
    float l_run[2] = {0.f, 0.f};              // this lane's share of the running sum

    // per-lane ldmatrix row offsets
    const int r16 = lane & 15, hi = lane >> 4;
    const uint32_t qa_row = q_s + (g * 16 + r16) * kRowBytes;
    const int key_b = (lane & 7) + (hi << 3);  // key row (within the warp's 16) of the S B-fragments

#pragma unroll 1
    for (int ch = 0; ch < nch; ++ch) {
        cp_async_wait1();
        __syncthreads();
        const uint32_t stage = st_s + (ch & 1) * kStageBytes;
        const uint8_t *vld = valid + (ch & 1) * kChunk;

        // ---- S = Q . K^T for 16 heads x 16 keys over 512 dims
        float s[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
        {
            const int krow = c * 16 + key_b;
            const uint32_t k_row = stage + krow * kRowBytes;
            const int sel = (lane >> 3) & 1;
#pragma unroll 8
            for (int kk = 0; kk < 32; ++kk) {
                uint32_t a[4], bb[4];
                ldsm_x4(qa_row + (((2 * kk + hi) ^ (lane & 7)) << 4), a);
                ldsm_x4(k_row + (((2 * kk + sel) ^ (lane & 7)) << 4), bb);
                mma16816<F16>(s[0], a, bb[0], bb[1]);
                mma16816<F16>(s[1], a, bb[2], bb[3]);
            }
        }

        // ---- online softmax over the chunk, shared by the group's 4 warps
        const int cc = lane & 3, rr = lane >> 2;
        float x[2][4];
        float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
            const int key = c * 16 + nt * 8 + 2 * cc;
            const bool v0 = vld[key] != 0, v1 = vld[key + 1] != 0;
            x[nt][0] = v0 ? s[nt][0] * p.scale_log2 : -INFINITY;
            x[nt][1] = v1 ? s[nt][1] * p.scale_log2 : -INFINITY;
            x[nt][2] = v0 ? s[nt][2] * p.scale_log2 : -INFINITY;
            x[nt][3] = v1 ? s[nt][3] * p.scale_log2 : -INFINITY;
            mx0 = fmaxf(mx0, fmaxf(x[nt][0], x[nt][1]));
            mx1 = fmaxf(mx1, fmaxf(x[nt][2], x[nt][3]));
        }
#pragma unroll
        for (int off = 1; off < 4; off <<= 1) {
            mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, off));
            mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, off));
        }
        float *red_g = red + g * 64;
        if (cc == 0) {
            red_g[c * 16 + rr] = mx0;
            red_g[c * 16 + rr + 8] = mx1;
        }
        group_bar(g, 128);
        float m_new[2], m_use[2], alpha[2];
#pragma unroll
        for (int h2 = 0; h2 < 2; ++h2) {
            const int row = rr + 8 * h2;
            float m = m_run[h2];
#pragma unroll
            for (int q = 0; q < 4; ++q) m = fmaxf(m, red_g[q * 16 + row]);
            m_new[h2] = m;
            m_use[h2] = m == -INFINITY ? 0.f : m;
            alpha[h2] = exp2f(m_run[h2] - m_use[h2]);  // 0 while nothing was valid yet
            m_run[h2] = m;
        }
        const uint32_t p_g = p_s + g * 16 * (kChunk * 2);
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
            const float p0 = exp2f(x[nt][0] - m_use[0]), p1 = exp2f(x[nt][1] - m_use[0]);
            const float p2 = exp2f(x[nt][2] - m_use[1]), p3 = exp2f(x[nt][3] - m_use[1]);
            l_run[0] = (nt == 0 ? l_run[0] * alpha[0] : l_run[0]) + p0 + p1;
            l_run[1] = (nt == 0 ? l_run[1] * alpha[1] : l_run[1]) + p2 + p3;
            const int key = c * 16 + nt * 8 + 2 * cc;
            const uint32_t off0 = rr * 128 + ((((key >> 3) ^ (rr & 7))) << 4) + ((key & 7) << 1);
            const uint32_t off1 = (rr + 8) * 128 + ((((key >> 3) ^ ((rr + 8) & 7))) << 4) + ((key & 7) << 1);
            asm volatile("st.shared.u32 [%0], %1;" ::"r"(p_g + off0), "r"(pack2<F16>(p0, p1)) : "memory");
            asm volatile("st.shared.u32 [%0], %1;" ::"r"(p_g + off1), "r"(pack2<F16>(p2, p3)) : "memory");
        }
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            o[i][0] *= alpha[0];
            o[i][1] *= alpha[0];
            o[i][2] *= alpha[1];
            o[i][3] *= alpha[1];
        }
        group_bar(g, 128);

        // ---- O += P . V for 16 heads x dims 128c..128c+127
        {
            const uint32_t pa_row = p_g + r16 * 128;
            const uint32_t v_row = stage + r16 * kRowBytes;
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
                uint32_t a[4];
                ldsm_x4(pa_row + (((2 * kk + hi) ^ (lane & 7)) << 4), a);
                const uint32_t vr = v_row + kk * 16 * kRowBytes;
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    uint32_t bb[4];
                    ldsm_x4_t(vr + (((c * 16 + 2 * j + hi) ^ (lane & 7)) << 4), bb);
                    mma16816<F16>(o[2 * j], a, bb[0], bb[1]);
                    mma16816<F16>(o[2 * j + 1], a, bb[2], bb[3]);
                }
            }
        }
        __syncthreads();
        if (ch + 2 < nch)
            gather_chunk<NT>(p, t, j_lo + (ch + 2) * kChunk, j_hi, stage, valid + (ch & 1) * kChunk);
        cp_async_commit();
    }

    // ---- the group's sums, then the results
    float lsum[2];
#pragma unroll
    for (int h2 = 0; h2 < 2; ++h2) {
        float v = l_run[h2];
        v += __shfl_xor_sync(0xffffffffu, v, 1);
        v += __shfl_xor_sync(0xffffffffu, v, 2);
        lsum[h2] = v;
    }
    __syncthreads();  // the red area is free again (also when there was no chunk)
    float *red_g = red + g * 64;
    const int cc = lane & 3, rr = lane >> 2;
    if (cc == 0) {
        red_g[c * 16 + rr] = lsum[0];
        red_g[c * 16 + rr + 8] = lsum[1];
    }
    group_bar(g, 128);
    float l_tot[2];
#pragma unroll
    for (int h2 = 0; h2 < 2; ++h2) {
        const int row = rr + 8 * h2;
        l_tot[h2] = red_g[row] + red_g[16 + row] + red_g[32 + row] + red_g[48 + row];
    }
    const int dim0 = c * 128 + 2 * cc;
    if (p.splits == 1) {
#pragma unroll
        for (int h2 = 0; h2 < 2; ++h2) {
            const int head = head0 + g * 16 + rr + 8 * h2;
            const float inv = l_tot[h2] > 0.f ? 1.f / l_tot[h2] : 0.f;
            float *dst = p.out + (t * p.Ha + head) * kDc + dim0;
#pragma unroll
            for (int i = 0; i < 16; ++i)
                *reinterpret_cast<float2 *>(dst + 8 * i) = make_float2(o[i][2 * h2] * inv, o[i][2 * h2 + 1] * inv);
            if (c == 0 && cc == 0)
                p.lse[t * p.Ha + head] =
                    l_tot[h2] > 0.f ? (m_run[h2] + log2f(l_tot[h2])) * kLn2 : -INFINITY;
        }
    } else {
#pragma unroll
        for (int h2 = 0; h2 < 2; ++h2) {
            const int head = head0 + g * 16 + rr + 8 * h2;
            const long long row = (t * p.splits + split) * p.Ha + head;
            float *dst = p.part_o + row * kDc + dim0;
#pragma unroll
            for (int i = 0; i < 16; ++i)
                *reinterpret_cast<float2 *>(dst + 8 * i) = make_float2(o[i][2 * h2], o[i][2 * h2 + 1]);
            if (c == 0 && cc == 0)
                *reinterpret_cast<float2 *>(p.part_ml + row * 2) = make_float2(m_run[h2], l_tot[h2]);
        }
    }
}

// Merge of the splits' partials: one CTA of 128 threads per (query, head),
// four dims per thread.
__global__ void __launch_bounds__(128) attn_combine_kernel(const float *part_o, const float *part_ml, float *out,
                                                            float *lse, int splits, int Ha) {
    const long long row = blockIdx.x;  // t * Ha + h
    const long long t = row / Ha, h = row % Ha;
    asm volatile("griddepcontrol.wait;" ::: "memory");
    float m = -INFINITY;
    for (int s = 0; s < splits; ++s) m = fmaxf(m, part_ml[((t * splits + s) * Ha + h) * 2]);
    const float m_use = m == -INFINITY ? 0.f : m;
    float l = 0.f;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int s = 0; s < splits; ++s) {
        const long long pr = (t * splits + s) * Ha + h;
        const float2 ml = *reinterpret_cast<const float2 *>(part_ml + pr * 2);
        const float w = exp2f(ml.x - m_use);
        l += w * ml.y;
        const float4 v = *reinterpret_cast<const float4 *>(part_o + pr * kDc + threadIdx.x * 4);
        acc.x += w * v.x;
        acc.y += w * v.y;
        acc.z += w * v.z;
        acc.w += w * v.w;
    }
    const float inv = l > 0.f ? 1.f / l : 0.f;
    *reinterpret_cast<float4 *>(out + row * kDc + threadIdx.x * 4) =
        make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv);
    if (threadIdx.x == 0) lse[row] = l > 0.f ? (m + log2f(l)) * kLn2 : -INFINITY;
}

}  // namespace attn
}  // namespace lid
