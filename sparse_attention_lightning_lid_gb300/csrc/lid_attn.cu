// lid_attn.cu -- host side of lid_sparse_attn: checks, the launch plan and the
// launches of the sparse-attention kernels (lid_attn.cuh).
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include <mutex>

#include "lid.h"
#include "lid_attn.cuh"
#include "lid_attn_tc.cuh"
#include "lid_internal.h"

namespace lid {
namespace {

struct AttnPlan {
    int path = 1;       // 1: warp-level MMA kernel, 2: tensor-core (tcgen05) kernel
    int G = 1;          // groups of 16 heads per CTA
    int head_blocks = 1;
    int splits = 1;
    int keys_per_split = 0;
    long long ctas = 0;
    long long ws_bytes = 0;
};

bool aligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

int check_shape(long long n_q, long long n_kv, int Ha, int Dc, int top_k) {
    if (n_q < 0 || n_kv < 0) return LID_ERR_INVALID_ARG;
    if (Dc != attn::kDc || (Ha != 16 && Ha != 32 && Ha != 64 && Ha != 128)) return LID_ERR_UNSUPPORTED;
    if (top_k < 1 || top_k > 2048 || n_kv > 2147483647ll) return LID_ERR_UNSUPPORTED;
    if (n_q > (2147483647ll / Ha) / 8) return LID_ERR_UNSUPPORTED;  // grid and row indices stay in range
    return LID_OK;
}

int make_plan(long long n_q, long long n_kv, int Ha, int top_k, const lid_attn_options *opt, int sm_count,
              AttnPlan *pl) {
    const int forced = opt ? opt->path : 0;
    if (forced < 0 || forced > 2) return LID_ERR_INVALID_ARG;
    // the tensor-core kernel takes 64 heads per CTA; it pays once there are
    // enough (query, 64-head block) pairs to spread over the SMs
    const bool tc_ok = Ha % attn::kTcHeads == 0 && n_kv > 0;
    if (forced == 2 && !tc_ok) return LID_ERR_UNSUPPORTED;
    const long long tc_blocks = n_q * (Ha / attn::kTcHeads);
    if (forced == 2 || (forced == 0 && tc_ok && tc_blocks * 4 >= sm_count)) {
        const int chunks = (top_k + attn::kTcKeys - 1) / attn::kTcKeys;
        int S;
        if (opt && opt->force_splits) {
            S = opt->force_splits < 1 ? 1 : (opt->force_splits > chunks ? chunks : opt->force_splits);
        } else if (tc_blocks >= sm_count) {
            S = 1;
        } else {
            const long long want = (sm_count + tc_blocks - 1) / tc_blocks;
            S = static_cast<int>(want < chunks ? want : chunks);
        }
        const int cps = (chunks + S - 1) / S;
        pl->path = 2;
        pl->G = attn::kTcHeads / 16;
        pl->head_blocks = Ha / attn::kTcHeads;
        pl->keys_per_split = cps * attn::kTcKeys;
        pl->splits = (top_k + pl->keys_per_split - 1) / pl->keys_per_split;
        pl->ctas = tc_blocks * pl->splits;
        pl->ws_bytes = pl->splits > 1 ? n_q * pl->splits * Ha * (attn::kDc * 4ll + 8) : 0;
        return LID_OK;
    }
    const int groups = Ha / 16;
    const int chunks = (top_k + attn::kChunk - 1) / attn::kChunk;
    int G;
    if (opt && opt->force_head_groups) {
        G = opt->force_head_groups;
        if ((G != 1 && G != 2 && G != 4) || groups % G) return LID_ERR_INVALID_ARG;
    } else {
        // all of a query's heads in one CTA (each gathered row serves them all)
        // when there are enough queries to fill the GPU; else one group per CTA
        G = groups < 4 ? groups : 4;
        if (n_q * (groups / G) < sm_count) G = 1;
    }
    const int hb = groups / G;
    const long long base = n_q * hb;
    int S;
    if (opt && opt->force_splits) {
        S = opt->force_splits < 1 ? 1 : (opt->force_splits > chunks ? chunks : opt->force_splits);
    } else if (base >= sm_count) {
        S = 1;
    } else {
        // split the selections until about one wave of CTAs
        const long long want = (sm_count + base - 1) / base;
        S = static_cast<int>(want < chunks ? want : chunks);
    }
    const int cps = (chunks + S - 1) / S;  // chunks per split
    pl->path = 1;
    pl->G = G;
    pl->head_blocks = hb;
    pl->keys_per_split = cps * attn::kChunk;
    pl->splits = (top_k + pl->keys_per_split - 1) / pl->keys_per_split;  // no empty split
    pl->ctas = base * pl->splits;
    pl->ws_bytes = pl->splits > 1 ? n_q * pl->splits * Ha * (attn::kDc * 4ll + 8) : 0;
    return LID_OK;
}

std::mutex g_attn_mutex;
unsigned long long g_attn_ctx[64] = {};
bool g_attn_attr[64][8] = {};

// Set a kernel's dynamic shared-memory limit once per context.
int ensure_smem_attr(const void *fn, int slot, int smem, int dev, unsigned long long ctx) {
    std::lock_guard<std::mutex> lock(g_attn_mutex);
    if (g_attn_ctx[dev] != ctx) {
        for (bool &b : g_attn_attr[dev]) b = false;
        g_attn_ctx[dev] = ctx;
    }
    if (!g_attn_attr[dev][slot]) {
        const cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess) return env_cuda_status(e);
        g_attn_attr[dev][slot] = true;
    }
    return LID_OK;
}

template <bool F16>
int launch_tc(const attn::Params &p, long long ctas, cudaStream_t st, int dev, unsigned long long ctx) {
    int rc;
    const int smem = attn::TcSmem::kTotal;
    if ((rc = ensure_smem_attr(reinterpret_cast<const void *>(attn::sparse_attn_tc_kernel<F16>), 6 + (F16 ? 1 : 0),
                               smem, dev, ctx)))
        return rc;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(ctas));
    cfg.blockDim = dim3(attn::kTcThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    return env_cuda_status(cudaLaunchKernelEx(&cfg, attn::sparse_attn_tc_kernel<F16>, p, kWaitLimitCycles));
}

template <int G, bool F16>
int launch_main(const attn::Params &p, long long ctas, cudaStream_t st, int dev, unsigned long long ctx) {
    constexpr int slot = (G == 1 ? 0 : G == 2 ? 1 : 2) * 2 + (F16 ? 1 : 0);
    const int smem = attn::Smem<G>::kTotal;
    const int rc = ensure_smem_attr(reinterpret_cast<const void *>(attn::sparse_attn_kernel<G, F16>), slot, smem, dev,
                                    ctx);
    if (rc) return rc;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(ctas));
    cfg.blockDim = dim3(128 * G);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    return env_cuda_status(cudaLaunchKernelEx(&cfg, attn::sparse_attn_kernel<G, F16>, p));
}

int launch_combine(const attn::Params &p, cudaStream_t st) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(p.n_q * p.Ha));
    cfg.blockDim = dim3(128);
    cfg.stream = st;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    return env_cuda_status(cudaLaunchKernelEx(&cfg, attn::attn_combine_kernel, (const float *)p.part_o,
                                              (const float *)p.part_ml, p.out, p.lse, p.splits, p.Ha));
}

int run_attn(const void *qa, const void *kv, const int32_t *idx, const float *sel_score, long long n_q,
             long long n_kv, int Ha, int Dc, int top_k, float scale, float *out, float *lse, void *workspace,
             long long workspace_bytes, cudaStream_t st, int dtype, const lid_attn_options *opt) {
    int rc = check_shape(n_q, n_kv, Ha, Dc, top_k);
    if (rc) return rc;
    if (dtype != LID_DTYPE_BF16 && dtype != LID_DTYPE_F16) return LID_ERR_INVALID_ARG;
    if (!isfinite(scale)) return LID_ERR_INVALID_ARG;
    if (n_q == 0) return LID_OK;
    if (!qa || !idx || !out || !lse || (n_kv > 0 && !kv)) return LID_ERR_INVALID_ARG;
    if (!aligned(qa, 16) || (kv && !aligned(kv, 16)) || !aligned(idx, 4) || !aligned(out, 16) ||
        !aligned(lse, 4) || (sel_score && !aligned(sel_score, 4)))
        return LID_ERR_INVALID_ARG;
    DeviceEnv env;
    if (env_device(&env)) return LID_ERR_CUDA;
    if (!env.sm103) return LID_ERR_UNSUPPORTED;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return LID_ERR_CUDA;
    AttnPlan pl;
    if ((rc = make_plan(n_q, n_kv, Ha, top_k, opt, env.sm_count, &pl))) return rc;

    attn::Params p = {};
    p.qa = static_cast<const uint16_t *>(qa);
    p.kv = static_cast<const uint16_t *>(kv);
    p.idx = idx;
    p.sel_score = sel_score;
    p.out = out;
    p.lse = lse;
    p.n_q = n_q;
    p.n_kv = n_kv;
    p.Ha = Ha;
    p.top_k = top_k;
    p.splits = pl.splits;
    p.keys_per_split = pl.keys_per_split;
    p.head_blocks = pl.head_blocks;
    p.scale_log2 = scale * attn::kLog2e;

    bool own_ws = false;
    void *ws = nullptr;
    if (pl.ws_bytes > 0) {
        if (workspace) {
            if (workspace_bytes < pl.ws_bytes) return LID_ERR_SCRATCH_TOO_SMALL;
            if (!aligned(workspace, 256)) return LID_ERR_INVALID_ARG;
            ws = workspace;
        } else {
            if (env_ws_alloc(&ws, static_cast<size_t>(pl.ws_bytes), st) != cudaSuccess) {
                cudaGetLastError();
                return LID_ERR_OOM;
            }
            own_ws = true;
        }
        p.part_o = static_cast<float *>(ws);
        p.part_ml = reinterpret_cast<float *>(static_cast<uint8_t *>(ws) + n_q * pl.splits * Ha * attn::kDc * 4ll);
    }
    const bool f16 = dtype == LID_DTYPE_F16;
    if (pl.path == 2) {
        rc = f16 ? launch_tc<true>(p, pl.ctas, st, dev, env.ctx_id) : launch_tc<false>(p, pl.ctas, st, dev, env.ctx_id);
    } else switch (pl.G * 2 + (f16 ? 1 : 0)) {
        case 2: rc = launch_main<1, false>(p, pl.ctas, st, dev, env.ctx_id); break;
        case 3: rc = launch_main<1, true>(p, pl.ctas, st, dev, env.ctx_id); break;
        case 4: rc = launch_main<2, false>(p, pl.ctas, st, dev, env.ctx_id); break;
        case 5: rc = launch_main<2, true>(p, pl.ctas, st, dev, env.ctx_id); break;
        case 8: rc = launch_main<4, false>(p, pl.ctas, st, dev, env.ctx_id); break;
        default: rc = launch_main<4, true>(p, pl.ctas, st, dev, env.ctx_id); break;
    }
    if (!rc && pl.splits > 1) rc = launch_combine(p, st);
    if (own_ws) {
        const int rc2 = env_cuda_status(cudaFreeAsync(ws, st));
        if (!rc) rc = rc2;
    }
    return rc;
}

}  // namespace

// The first device-side error code this translation unit's kernels recorded
// (their module's own error word); reset != 0 clears it. Synchronous.
int attn_device_error(int reset) {
    int v = 0;
    if (cudaMemcpyFromSymbol(&v, g_dev_error, sizeof(int)) != cudaSuccess) return -1;
    if (reset && v) {
        const int zero = 0;
        cudaMemcpyToSymbol(g_dev_error, &zero, sizeof(int));
    }
    return v;
}

}  // namespace lid

extern "C" {

int lid_sparse_attn(const void *qa, const void *kv, const int32_t *idx, const float *sel_score, int64_t n_q,
                    int64_t n_kv, int Ha, int Dc, int top_k, float scale, float *out, float *lse, void *workspace,
                    int64_t workspace_bytes, void *stream, int dtype, const lid_attn_options *opt) {
    return lid::run_attn(qa, kv, idx, sel_score, n_q, n_kv, Ha, Dc, top_k, scale, out, lse, workspace,
                         workspace_bytes, static_cast<cudaStream_t>(stream), dtype, opt);
}

int lid_sparse_attn_plan(int64_t n_q, int64_t n_kv, int Ha, int Dc, int top_k, const lid_attn_options *opt,
                         lid_attn_plan_info *info) {
    if (!info) return LID_ERR_INVALID_ARG;
    int rc = lid::check_shape(n_q, n_kv, Ha, Dc, top_k);
    if (rc) return rc;
    lid::DeviceEnv env;
    if (lid::env_device(&env)) return LID_ERR_CUDA;
    lid::AttnPlan pl;
    if ((rc = lid::make_plan(n_q, n_kv, Ha, top_k, opt, env.sm_count, &pl))) return rc;
    info->path = pl.path;
    info->head_groups = pl.G;
    info->splits = pl.splits;
    info->keys_per_split = pl.keys_per_split;
    info->ctas = pl.ctas;
    info->workspace_bytes = pl.ws_bytes;
    return LID_OK;
}

}  // extern "C"
