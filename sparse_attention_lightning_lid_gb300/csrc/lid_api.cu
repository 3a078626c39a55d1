// lid_api.cu -- host side of the lightning-indexer top-k library: argument
// validation, launch planning, tensor maps, workspace and launches.
// The C ABI is declared in include/lid.h.
#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <mutex>

#include "lid.h"
#include "lid_internal.h"
#include "lid_kernels.cuh"
#include "lid_stream.cuh"

namespace lid {
namespace {

constexpr int kMaxDevices = 64;

struct DeviceInfo {
    bool ready = false;
    unsigned long long ctx_id = 0;  // the context these cached handles and addresses belong to
    cudaMemPool_t pool = nullptr;  // workspace pool that keeps its memory mapped
    bool sm103 = false;
    int sm_count = 0;
    int smem_optin = 0;
    bool attr_set[12] = {};    // scoring kernels H = 8, 16, 32, 64; merge; one-launch kernels H = 8 .. 64;
                               // single-query kernels H = 16, 32, 64
    int coop_blocks[7] = {};   // resident CTAs per SM of the one-launch kernels (0: not yet asked)
    uint32_t coop_smem[7] = {}; // ... for this much dynamic shared memory
    // host-buffer calls (g_host_mutex): the stream their input copies run on, per
    // call slot (call number mod 2) the end of its copies and the end of the call
    cudaStream_t copy_stream = nullptr;
    cudaEvent_t host_copied[2] = {};
    cudaEvent_t host_done[2] = {};
    unsigned long long host_calls = 0;
};

std::mutex g_mutex;
std::mutex g_host_mutex;  // host-buffer calls enqueue one at a time (their copy stream and events)
DeviceInfo g_dev[kMaxDevices];

// Group-barrier slots of the one-launch path: counters that start at zero (the
// array is zero when the module loads) and that each launch leaves at zero
// (its last CTA per group clears them), so no memset is needed per call. A
// slot is never used by two launches that can overlap: eager calls use the
// slot of their stream (calls on one stream are ordered), and a call recorded
// into a graph gets a slot of its own. When the slots run out, the counters
// go back to the workspace, zeroed by a memset on the stream.
constexpr int kCtrlStreamSlots = 256;
constexpr int kCtrlSlots = 1024;
constexpr int kCtrlWords = 2 * 80;  // bar and done counters of up to 80 query groups
static __device__ unsigned g_ctrl[kCtrlSlots][kCtrlWords];
struct CtrlState {
    unsigned *base = nullptr;  // device address of g_ctrl (nullptr: not looked up / failed)
    bool looked_up = false;
    // streams by their ID (cudaStreamGetId: unique for the life of the process,
    // never reused by a later stream, and the calling thread's own for
    // cudaStreamPerThread), so two streams that can overlap never share a slot
    unsigned long long stream_of[kCtrlStreamSlots] = {};
    int n_stream = 0;
    int next_graph = kCtrlStreamSlots;
};
CtrlState g_ctrl_state[kMaxDevices];
void *g_static_scratch_ptr[kMaxDevices] = {};  // device address of the static scratch (see run_static)
thread_local cudaError_t g_last_cuda_error = cudaSuccess;

// Turn a CUDA result into a status, remembering the failure for lid_last_cuda_error().
int cuda_status(cudaError_t e) {
    if (e == cudaSuccess) return LID_OK;
    g_last_cuda_error = e;
    return LID_ERR_CUDA;
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                  const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn g_encode = nullptr;
typedef CUresult (*CtxGetCurrentFn)(CUcontext *);
typedef CUresult (*CtxGetIdFn)(CUcontext, unsigned long long *);
CtxGetCurrentFn g_ctx_current = nullptr;
CtxGetIdFn g_ctx_id = nullptr;

template <class F>
bool driver_fn(const char *name, F *out) {
    if (*out) return true;
    void *fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion(name, &fn, 12000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess || fn == nullptr)
        return false;
    *out = reinterpret_cast<F>(fn);
    return true;
}

// ID of the calling thread's current context (unique for the process's life:
// a device reset makes a new context with a new ID).
int current_ctx_id(unsigned long long *id) {
    if (!driver_fn("cuCtxGetCurrent", &g_ctx_current) || !driver_fn("cuCtxGetId", &g_ctx_id)) return LID_ERR_CUDA;
    CUcontext ctx = nullptr;
    if (g_ctx_current(&ctx) != CUDA_SUCCESS) return LID_ERR_CUDA;
    if (ctx == nullptr) {
        // no context yet on this thread (so no capture either): make the current
        // device's primary context current
        if (cudaFree(nullptr) != cudaSuccess || g_ctx_current(&ctx) != CUDA_SUCCESS || ctx == nullptr) {
            cudaGetLastError();
            return LID_ERR_CUDA;
        }
    }
    return g_ctx_id(ctx, id) == CUDA_SUCCESS ? LID_OK : LID_ERR_CUDA;
}

int device_info(DeviceInfo **out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return LID_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_mutex);
    unsigned long long cid = 0;
    if (current_ctx_id(&cid)) return LID_ERR_CUDA;
    DeviceInfo &d = g_dev[dev];
    if (d.ready && d.ctx_id != cid) {
        // the device was reset since the handles were cached: they (the pool, the
        // kernels' attributes, the static arrays' addresses) belong to a context
        // that is gone, so look everything up again
        d = DeviceInfo();
        g_ctrl_state[dev] = CtrlState();
        g_static_scratch_ptr[dev] = nullptr;
    }
    if (!d.ready) {
        d.ctx_id = cid;
        int major = 0, minor = 0;
        if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&d.sm_count, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&d.smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess)
            return LID_ERR_CUDA;
        d.sm103 = (major == 10 && minor == 3);
        // A pool of our own whose memory stays mapped between calls, so that a
        // call's workspace does not come back freshly mapped (and TLB-cold)
        // after every synchronisation; without it, the device's default pool.
        cudaMemPoolProps props = {};
        props.allocType = cudaMemAllocationTypePinned;
        props.location.type = cudaMemLocationTypeDevice;
        props.location.id = dev;
        if (cudaMemPoolCreate(&d.pool, &props) == cudaSuccess) {
            uint64_t keep = ~0ull;
            cudaMemPoolSetAttribute(d.pool, cudaMemPoolAttrReleaseThreshold, &keep);
        } else {
            cudaGetLastError();
            d.pool = nullptr;
        }
        d.ready = true;
    }
    if (!driver_fn("cuTensorMapEncodeTiled", &g_encode)) return LID_ERR_CUDA;
    *out = &d;
    return LID_OK;
}

// Stream-ordered workspace: our pool outside stream capture; inside a capture
// a plain cudaMallocAsync, which becomes a graph memory node.
cudaError_t ws_alloc(void **ptr, size_t bytes, cudaStream_t st, const DeviceInfo &dev) {
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    const cudaError_t e = cudaStreamIsCapturing(st, &cs);
    if (e != cudaSuccess) return e;
    if (dev.pool != nullptr && cs == cudaStreamCaptureStatusNone) return cudaMallocFromPoolAsync(ptr, bytes, dev.pool, st);
    return cudaMallocAsync(ptr, bytes, st);
}

// Every workspace starts with this many bytes for the one-launch path's
// group-barrier counters; nothing else ever writes them, so a workspace that
// is zero there stays usable for any later call (each launch leaves them zero).
constexpr long long kCounterBytes = 1024;

int next_pow2(int x) {
    int p = 1;
    while (p < x) p <<= 1;
    return p;
}

int round_up(int x, int m) { return (x + m - 1) / m * m; }

struct Plan {
    int qg, N, threads, n_groups, n_tiles, splits, tps, kstages, acc_stages, cap, P, tmem_cols;
    uint32_t smem;
    long long ws_bytes;
    long long off_qbound;  // (split lists) the per-query certified bounds, zeroed per call; 0: none
    int merge_cap;
    uint32_t merge_smem;
    bool fused;  // the split merge runs inside the scoring launch (cooperative)
    bool single; // ... by the single-query kernel (one query per CTA, every key of a CTA in its buffer)
    bool early;    // (fused, one query per group) steps A-B overlap the streaming
    int tilepar;   // one query per CTA and no cut possible: this many epilogue groups take tiles in turn
    int f_cap, f_pub, f_regcap;
    long long off_count, off_hist, off_stats, off_cand, off_reg;  // workspace offsets of the one-launch path
};


bool aligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

int validate_shape(long long n_q, long long n_kv, int H, int D, int top_k) {
    if (n_q < 0 || n_kv < 0) return LID_ERR_INVALID_ARG;
    if (!(H == 8 || H == 16 || H == 32 || H == 64)) return LID_ERR_UNSUPPORTED;
    if (!(D == 64 || D == 128)) return LID_ERR_UNSUPPORTED;
    if (top_k < 1 || top_k > 2048) return LID_ERR_UNSUPPORTED;
    if (n_kv > 0x7FFFFFFFll) return LID_ERR_UNSUPPORTED;
    if (n_q * H > 0x7FFFFFFFll) return LID_ERR_UNSUPPORTED;
    return LID_OK;
}

// Estimated run time of the scoring kernel plus merge, in units of one
// tile's work on one SM, for `splits` key splits.
double plan_cost(const Plan &p, long long n_q, int sms, int splits, int *tps_out, int *eff_out) {
    const int tps = (p.n_tiles + splits - 1) / splits;
    const int eff = (p.n_tiles + tps - 1) / tps;
    const long long ctas = static_cast<long long>(p.n_groups) * eff;
    const long long waves = (ctas + sms - 1) / sms;
    const double per_cta = tps + 3.0;  // set-up, final select, sort and write ~ 3 tiles
    double cost = static_cast<double>(waves) * per_cta;
    if (eff > 1) {
        const double rounds = static_cast<double>(eff) * p.P / kMergeThreads;
        cost += static_cast<double>((n_q + sms - 1) / sms) * (2.0 + 0.05 * rounds);
    }
    *tps_out = tps;
    *eff_out = eff;
    return cost;
}

int make_plan(long long n_q, long long n_kv, int H, int D, int top_k, const lid_options *opt,
              const DeviceInfo &dev, Plan *out, bool ranges = false) {
    Plan p{};
    p.P = next_pow2(top_k);
    p.n_tiles = static_cast<int>((n_kv + kBM - 1) / kBM);
    const int qg_full = 256 / H;
    const int qg_min = 16 / H > 1 ? 16 / H : 1;
    int qg;
    if (opt && opt->force_qg) {
        qg = opt->force_qg;
        if (qg < 1 || (qg & (qg - 1)) != 0 || qg * H < 16 || qg * H > 256) return LID_ERR_INVALID_ARG;
    } else if (ranges && n_q <= 8) {
        // a few rows with their own key ranges (multi-sequence decode): one row
        // per CTA, so that each CTA streams only the tiles of its row's range
        qg = qg_min;
    } else {
        const int want = next_pow2(static_cast<int>(n_q < qg_full ? (n_q > 0 ? n_q : 1) : qg_full));
        qg = want < qg_min ? qg_min : (want > qg_full ? qg_full : want);
    }
    // a buffer holds top_k keys plus one tile of new candidates
    const int min_cap = round_up(top_k + kBM, kBM);
    for (;;) {
        p.qg = qg;
        p.N = qg * H;
        p.threads = kScoreThreads;
        p.acc_stages = 512 / p.N < kMaxAccStages ? 512 / p.N : kMaxAccStages;
        p.tmem_cols = next_pow2(p.acc_stages * p.N < 32 ? 32 : p.acc_stages * p.N);
        const int pref_cap = min_cap > round_up(2 * top_k + kBM, kBM) ? min_cap : round_up(2 * top_k + kBM, kBM);
        int best_ks = 0, best_cap = 0;
        const int ks_hi = (opt && opt->force_kstages) ? opt->force_kstages : 6;
        const int ks_lo = (opt && opt->force_kstages) ? opt->force_kstages : 2;
        if (ks_hi < 2 || ks_hi > kMaxKStages) return LID_ERR_INVALID_ARG;
        for (int pass = 0; pass < 2 && best_ks == 0; ++pass) {
            for (int ks = ks_hi; ks >= ks_lo; --ks) {
                const SmemLayout L0 = smem_layout(D, p.N, qg, H, ks, 0);
                const long long avail = static_cast<long long>(dev.smem_optin) - L0.total;
                if (avail <= 0) continue;
                int cap = static_cast<int>(avail / (8ll * qg)) / kBM * kBM;
                if (cap > kMaxCap) cap = kMaxCap;
                // the final sorts borrow the K stages as scratch
                const uint32_t fs = final_scratch_bytes(qg, L0.stage_bytes * static_cast<uint32_t>(ks));
                if (fs < static_cast<uint32_t>(kFinalScratchBytes)) continue;
                if (cap >= (pass == 0 ? pref_cap : min_cap)) {
                    best_ks = ks;
                    best_cap = cap;
                    break;
                }
            }
        }
        if (best_ks) {
            p.kstages = best_ks;
            p.cap = best_cap;
            break;
        }
        if ((opt && opt->force_qg) || qg <= qg_min) return LID_ERR_UNSUPPORTED;
        qg >>= 1;
    }
    p.smem = smem_layout(D, p.N, p.qg, H, p.kstages, p.cap).total;
    p.n_groups = static_cast<int>((n_q + p.qg - 1) / p.qg);
    if (p.n_tiles == 0) {
        p.splits = 1;
        p.tps = 0;
    } else if (opt && opt->force_splits) {
        int s = opt->force_splits < 1 ? 1 : (opt->force_splits > p.n_tiles ? p.n_tiles : opt->force_splits);
        if (s > kMaxSplits) s = kMaxSplits;
        p.tps = (p.n_tiles + s - 1) / s;
        p.splits = (p.n_tiles + p.tps - 1) / p.tps;
    } else {
        double best = 1e300;
        const int smax = p.n_tiles < kMaxSplits ? p.n_tiles : kMaxSplits;
        for (int s = 1; s <= smax; ++s) {
            int tps, eff;
            const double c = plan_cost(p, n_q, dev.sm_count, s, &tps, &eff);
            if (c < best * 0.999) {
                best = c;
                p.tps = tps;
                p.splits = eff;
            }
        }
    }
    p.ws_bytes = p.splits > 1 ? kCounterBytes + n_q * static_cast<long long>(p.splits) * top_k * 8ll : 0;
    if (static_cast<size_t>(dev.smem_optin) < kMergeSmem || top_k + kMergeThreads > kMergeCap)
        return LID_ERR_UNSUPPORTED;
    // One launch instead of split lists + merge when all CTAs of a query group
    // fit on the GPU at once (one CTA per SM): by default wherever the plan
    // splits the keys and no split count is forced.
    const int path = opt ? opt->path : 0;
    if (path < 0 || path > 3) return LID_ERR_INVALID_ARG;
    p.fused = false;
    const bool want = path >= 2 || (path == 0 && p.splits > 1 && !(opt && opt->force_splits));
    p.early = false;
    p.f_pub = 0;
    if (want && p.n_tiles > 0) {
        const int per_group = dev.sm_count / p.n_groups;
        int s = (opt && opt->force_splits) ? opt->force_splits : per_group;
        s = s < 1 ? 1 : (s > p.n_tiles ? p.n_tiles : s);
        const int tps = (p.n_tiles + s - 1) / s;
        const int eff = (p.n_tiles + tps - 1) / tps;
        // one query per group (H >= 32): group 0 streams while the idle epilogue
        // groups run steps A-B; their scratch takes shared memory from the K stages
        int ks = p.kstages, cap = p.cap;
        bool early = p.qg == 1 && H >= 32 && tps >= 2;
        if (early) {
            const int min_cap = round_up(top_k + kBM, kBM);
            bool fit = false;
            // with visible ranges a CTA's keys are often few enough to all fit a larger
            // buffer (then its epilogue groups take the tiles in turn, no cut): three K
            // stages, the rest of shared memory for the buffer
            const int ks_top = ranges && p.kstages > 3 ? 3 : p.kstages;
            const int cap_max = ranges ? kMaxCapRanges : kMaxCap;
            for (ks = ks_top; ks >= 2; --ks) {
                const SmemLayout L0 = smem_layout(D, p.N, p.qg, H, ks, 0, kEarlyBytes);
                const long long avail = static_cast<long long>(dev.smem_optin) - L0.total;
                if (avail <= 0) continue;
                cap = static_cast<int>(avail / (8ll * p.qg)) / kBM * kBM;
                if (cap > cap_max) cap = cap_max;
                if (cap >= min_cap) {
                    fit = true;
                    break;
                }
            }
            if (!fit) {
                early = false;
                ks = p.kstages;
                cap = p.cap;
            }
        }
        const long long kst = static_cast<long long>(smem_layout(D, p.N, p.qg, H, ks, 0).stage_bytes) * ks;
        const long long room = kst - kFusedHdr;
        // shared scratch of the tail: unit maxima, or certificates + bin members + histograms
        const long long need_a = static_cast<long long>(p.qg) * 128 * 8;
        const long long need_b = 2048;  // one warp's bins for the bound step
        const long long need = need_a > need_b ? need_a : need_b;
        const int f_cap = room / 8 < kFusedCapMax ? static_cast<int>(room / 8) : kFusedCapMax;
        const bool regs_ok = eff <= 32 * kBoundVPL;  // a warp holds one level's certificates
        if (eff >= 2 && eff <= per_group && room >= need && f_cap >= 2 * top_k && regs_ok) {
            auto r256 = [](long long x) { return (x + 255) / 256 * 256; };
            p.fused = true;
            p.early = early;
            p.f_regcap = 0;
            if (early) {
                p.kstages = ks;
                p.cap = cap;
                // certificates from the first ~4/7 of the tiles (later: a tighter bound, less
                // time to agree on it before the stream ends)
                const int pub = (opt && opt->early_tiles > 0) ? opt->early_tiles : (tps * 4) / 7;
                p.f_pub = pub < 1 ? 1 : (pub > tps ? tps : pub);
                // per-split regions for the keys >= the bound: room for three to six times
                // a split's even share of 2 top_k candidates (an overflow falls back to the
                // gather through the candidate list)
                int rc = next_pow2(static_cast<int>((6ll * top_k + eff - 1) / eff)) - 1;
                if (rc < 31) rc = 31;
                if (2ll * eff * (rc + 1) <= kst / 8) p.f_regcap = rc;
            }
            p.splits = eff;
            p.tps = tps;
            p.f_cap = f_cap;
            p.off_count = kCounterBytes;  // (2 n_groups counters at the head: n_groups <= 76 here)
            p.off_hist = p.off_count + r256(n_q * kFusedAttempts * 4ll);
            p.off_stats = p.off_hist + r256(kFusedRounds * n_q * 256 * 4ll);
            p.off_cand = p.off_stats + r256(n_q * eff * kFusedLevels * 8ll);
            p.off_reg = p.off_cand + r256(n_q * static_cast<long long>(f_cap) * 8);
            p.ws_bytes = p.off_reg + n_q * static_cast<long long>(eff) * (p.f_regcap + 1) * 8;
        } else if (path >= 2) {
            return LID_ERR_UNSUPPORTED;
        }
    } else if (path >= 2) {
        return LID_ERR_UNSUPPORTED;
    }
    p.single = false;
    if (p.fused && p.qg == 1 && !ranges && H >= 16 && path != 3) {
        // The single-query kernel: one query per CTA, every key of a CTA fits its
        // candidate buffer (no cut), and its K stages hold the tail's two copies of
        // the per-split regions. Stages sized for 16-bit operands (as above).
        const int cap1 = p.tps * kBM;
        for (int ks = 6; ks >= 2 && !p.single; --ks) {
            const SQLayout L = sq_layout(D, H, 2, ks, cap1);
            const long long room = static_cast<long long>(L.stage) * ks;
            if (L.total <= static_cast<uint32_t>(dev.smem_optin) && room >= 2ll * p.splits * kSQRegion * 8) {
                auto r256 = [](long long x) { return (x + 255) / 256 * 256; };
                p.single = true;
                p.kstages = ks;
                p.cap = cap1;
                p.threads = kSQThreads;
                p.tmem_cols = next_pow2(kSQAcc * H < 32 ? 32 : kSQAcc * H);
                p.acc_stages = kSQAcc;
                p.early = false;
                p.tilepar = 0;
                const int pub = (opt && opt->early_tiles > 0) ? opt->early_tiles : (p.tps * 4) / 7;
                p.f_pub = pub < 1 ? 1 : (pub > p.tps ? p.tps : pub);
                p.f_regcap = kSQRegion - 1;
                p.f_cap = p.splits * top_k;  // the overflow list: at most top_k keys from each split
                p.off_count = kCounterBytes;
                p.off_stats = p.off_count + r256(n_q * 4ll);
                p.off_reg = p.off_stats + r256(n_q * p.splits * kFusedLevels * 8ll);
                p.off_cand = p.off_reg + r256(n_q * p.splits * kSQRegion * 8ll);
                p.ws_bytes = p.off_cand + n_q * static_cast<long long>(p.f_cap) * 8;
                p.smem = L.total;
            }
        }
    }
    p.merge_cap = kMergeCap;
    p.merge_smem = static_cast<uint32_t>(kMergeSmem);
    if (!p.single) p.smem = smem_layout(D, p.N, p.qg, H, p.kstages, p.cap, p.early ? kEarlyBytes : 0u).total;
    // one query per CTA whose keys all fit the candidate buffer (no cut): the
    // epilogue groups take tiles in turn, two of them when the other two run
    // the early steps
    p.tilepar = (!p.single && p.qg == 1 && p.n_tiles > 0 && static_cast<long long>(p.tps) * kBM + kBM <= p.cap)
                    ? (p.early ? 2 : 4)
                    : 0;
    p.off_qbound = 0;
    if (!p.fused && p.splits > 1) {
        p.off_qbound = (p.ws_bytes + 255) / 256 * 256;
        p.ws_bytes = p.off_qbound + n_q * 8ll;
    }
    *out = p;
    return LID_OK;
}

// Record a caller's timing event; inside a stream capture it must become an
// external event node so that it is really recorded at replay.
int record_event(void *ev, cudaStream_t st) {
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(st, &cs) != cudaSuccess) return LID_ERR_CUDA;
    const unsigned flags = cs == cudaStreamCaptureStatusActive ? cudaEventRecordExternal : cudaEventRecordDefault;
    return cuda_status(cudaEventRecordWithFlags(static_cast<cudaEvent_t>(ev), st, flags));
}

// Row-major [outer][inner] of esize-byte elements, boxes of 128 bytes by
// box_outer rows, 128-byte swizzle (the MMA operand layout).
int encode_2d(CUtensorMap *m, const void *base, unsigned long long inner, unsigned long long outer, int esize,
              unsigned box_outer) {
    const cuuint64_t dims[2] = {inner, outer};
    const cuuint64_t strides[1] = {inner * static_cast<unsigned long long>(esize)};
    const cuuint32_t box[2] = {128u / static_cast<unsigned>(esize), box_outer};
    const cuuint32_t estr[2] = {1, 1};
    const CUtensorMapDataType ty = esize == 1 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_UINT16;
    const CUresult r = g_encode(m, ty, 2, const_cast<void *>(base), dims, strides, box,
                                estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                                CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? LID_OK : LID_ERR_CUDA;
}

template <int H, bool FUSED>
int launch_score(const CUtensorMap &tmk, const CUtensorMap &tmq, const ScoreParams &sp, const Plan &p,
                 DeviceInfo &dev, int hslot, cudaStream_t st) {
    auto kern = score_select_kernel<H, FUSED>;
    const int slot = FUSED ? 5 + hslot : hslot;
    if (!dev.attr_set[slot]) {
        int rc = cuda_status(cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, dev.smem_optin));
        // the same (all-shared) carveout as the merge, so no reconfiguration between them
        if (!rc)
            rc = cuda_status(cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout,
                                                  cudaSharedmemCarveoutMaxShared));
        if (rc) return rc;
        dev.attr_set[slot] = true;
    }
    const unsigned grid = static_cast<unsigned>(p.n_groups) * static_cast<unsigned>(p.splits);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(static_cast<unsigned>(p.threads));
    cfg.dynamicSmemBytes = p.smem;
    cfg.stream = st;
    // a programmatic dependent of whatever precedes it on the stream: the
    // kernel's prologue (barriers, tensor memory) overlaps that work's tail, and
    // it reads no global memory before griddepcontrol.wait
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (FUSED) {
        // the group barriers need every CTA resident: a cooperative launch, which
        // the runtime refuses rather than run partly
        int nb = 0;
        {
            std::lock_guard<std::mutex> lock(g_mutex);
            if (dev.coop_smem[hslot] == p.smem) nb = dev.coop_blocks[hslot];
        }
        if (nb == 0) {
            const int rc = cuda_status(cudaOccupancyMaxActiveBlocksPerMultiprocessor(&nb, kern, p.threads, p.smem));
            if (rc) return rc;
            std::lock_guard<std::mutex> lock(g_mutex);
            dev.coop_blocks[hslot] = nb;
            dev.coop_smem[hslot] = p.smem;
        }
        if (static_cast<long long>(grid) > static_cast<long long>(nb) * dev.sm_count) return LID_ERR_UNSUPPORTED;
        attr[1].id = cudaLaunchAttributeCooperative;
        attr[1].val.cooperative = 1;
        cfg.numAttrs = 2;
    }
    return cuda_status(cudaLaunchKernelEx(&cfg, kern, tmk, tmq, sp));
}

// The single-query kernel (H >= 16): cooperative, programmatic dependent.
template <int H>
int launch_single(const CUtensorMap &tmk, const CUtensorMap &tmq, const ScoreParams &sp, const Plan &p,
                  DeviceInfo &dev, int hslot, cudaStream_t st) {
    auto kern = stream_select_kernel<H>;
    const int slot = 9 + hslot - 1;  // H = 16, 32, 64 -> hslot 1, 2, 3
    if (!dev.attr_set[slot]) {
        int rc = cuda_status(cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, dev.smem_optin));
        if (!rc)
            rc = cuda_status(cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout,
                                                  cudaSharedmemCarveoutMaxShared));
        if (rc) return rc;
        dev.attr_set[slot] = true;
    }
    const unsigned grid = static_cast<unsigned>(p.n_groups) * static_cast<unsigned>(p.splits);
    const int cslot = 4 + hslot - 1;
    int nb = 0;
    {
        std::lock_guard<std::mutex> lock(g_mutex);
        if (dev.coop_smem[cslot] == p.smem) nb = dev.coop_blocks[cslot];
    }
    if (nb == 0) {
        const int rc = cuda_status(cudaOccupancyMaxActiveBlocksPerMultiprocessor(&nb, kern, p.threads, p.smem));
        if (rc) return rc;
        std::lock_guard<std::mutex> lock(g_mutex);
        dev.coop_blocks[cslot] = nb;
        dev.coop_smem[cslot] = p.smem;
    }
    if (static_cast<long long>(grid) > static_cast<long long>(nb) * dev.sm_count) return LID_ERR_UNSUPPORTED;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(static_cast<unsigned>(p.threads));
    cfg.dynamicSmemBytes = p.smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    attr[1].id = cudaLaunchAttributeCooperative;
    attr[1].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    return cuda_status(cudaLaunchKernelEx(&cfg, kern, tmk, tmq, sp));
}

template <int H>
int launch_score_h(const CUtensorMap &tmk, const CUtensorMap &tmq, const ScoreParams &sp, const Plan &p,
                   DeviceInfo &dev, int hslot, cudaStream_t st) {
    if constexpr (H >= 16) {
        if (p.single) return launch_single<H>(tmk, tmq, sp, p, dev, hslot, st);
    }
    return p.fused ? launch_score<H, true>(tmk, tmq, sp, p, dev, hslot, st)
                   : launch_score<H, false>(tmk, tmq, sp, p, dev, hslot, st);
}

// Plans of recent shapes: the planner searches every split count, which
// would cost more host time per call than a decode step takes on the GPU. A
// plan is a pure function of its key (and of the device, whose entry holds
// the cache), so the cache only saves time.
struct PlanKey {
    long long n_q, n_kv;
    int H, D, top_k, ranges, force_splits, force_qg, force_kstages, path, early_tiles;
    bool operator==(const PlanKey &o) const {
        return n_q == o.n_q && n_kv == o.n_kv && H == o.H && D == o.D && top_k == o.top_k && ranges == o.ranges &&
               force_splits == o.force_splits && force_qg == o.force_qg && force_kstages == o.force_kstages &&
               path == o.path && early_tiles == o.early_tiles;
    }
};
constexpr int kPlanCache = 32;
struct PlanCache {
    PlanKey key[kPlanCache];
    Plan plan[kPlanCache];
    int n = 0, next = 0;
    unsigned long long ctx_id = 0;  // the context of the device entry the plans were made for
};
PlanCache g_plan_cache[kMaxDevices];

int cached_plan(long long n_q, long long n_kv, int H, int D, int top_k, const lid_options *opt, DeviceInfo &dev,
                Plan *out, bool ranges) {
    PlanKey k{n_q, n_kv, H, D, top_k, ranges ? 1 : 0, opt ? opt->force_splits : 0, opt ? opt->force_qg : 0,
              opt ? opt->force_kstages : 0, opt ? opt->path : 0, opt ? opt->early_tiles : 0};
    const int d = static_cast<int>(&dev - g_dev);
    {
        std::lock_guard<std::mutex> lock(g_mutex);
        PlanCache &c = g_plan_cache[d];
        if (c.ctx_id != dev.ctx_id) {
            c.n = c.next = 0;
            c.ctx_id = dev.ctx_id;
        }
        for (int i = 0; i < c.n; ++i)
            if (c.key[i] == k) {
                *out = c.plan[i];
                return LID_OK;
            }
    }
    const int rc = make_plan(n_q, n_kv, H, D, top_k, opt, dev, out, ranges);
    if (rc) return rc;
    std::lock_guard<std::mutex> lock(g_mutex);
    PlanCache &c = g_plan_cache[d];
    c.key[c.next] = k;
    c.plan[c.next] = *out;
    c.next = (c.next + 1) % kPlanCache;
    if (c.n < kPlanCache) ++c.n;
    return LID_OK;
}

// Checks shared by the entry points; fills *dev and *p.
int prepare(const void *q, const void *k, const float *w, const void *mask, long long n_q, long long n_kv, int H,
            int D, int top_k, const int32_t *out_idx, const float *out_score, int dtype, const lid_options *opt,
            DeviceInfo **dev, Plan *p, const int32_t *row_lo = nullptr, const int32_t *row_hi = nullptr,
            const float *q_scale = nullptr, const float *k_scale = nullptr) {
    int rc = validate_shape(n_q, n_kv, H, D, top_k);
    if (rc) return rc;
    if (dtype != LID_DTYPE_BF16 && dtype != LID_DTYPE_F16 && dtype != LID_DTYPE_E4M3) return LID_ERR_INVALID_ARG;
    // 8-bit rows of 128 elements fill one 128-byte swizzle span; shorter rows would need another layout
    if (dtype == LID_DTYPE_E4M3 && D != 128) return LID_ERR_UNSUPPORTED;
    if (n_q == 0) return LID_OK;
    if (dtype == LID_DTYPE_E4M3 && n_kv > 0 &&
        (!q_scale || !k_scale || !aligned(q_scale, 4) || !aligned(k_scale, 4)))
        return LID_ERR_INVALID_ARG;
    if (!out_idx || !out_score || !aligned(out_idx, 4) || !aligned(out_score, 4)) return LID_ERR_INVALID_ARG;
    if (n_kv > 0) {
        if (!q || !k || !w) return LID_ERR_INVALID_ARG;
        if (!aligned(q, 16) || !aligned(k, 16) || !aligned(w, 4) || (mask && !aligned(mask, 2)))
            return LID_ERR_INVALID_ARG;
    }
    if ((row_lo == nullptr) != (row_hi == nullptr)) return LID_ERR_INVALID_ARG;
    if (row_lo && (mask || !aligned(row_lo, 4) || !aligned(row_hi, 4))) return LID_ERR_INVALID_ARG;
    rc = device_info(dev);
    if (rc) return rc;
    if (!(*dev)->sm103) return LID_ERR_UNSUPPORTED;
    return cached_plan(n_q, n_kv, H, D, top_k, opt, **dev, p, row_lo != nullptr);
}

// Counters for one fused launch on `st` (n_groups groups): a self-clearing
// slot, or nullptr (then the caller zeroes workspace counters with a memset).
unsigned *ctrl_slot(cudaStream_t st, int n_groups) {
    if (n_groups * 2 > kCtrlWords) return nullptr;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(st, &cs) != cudaSuccess) {
        cudaGetLastError();
        return nullptr;
    }
    unsigned long long sid = 0;
    if (cs != cudaStreamCaptureStatusActive && cudaStreamGetId(st, &sid) != cudaSuccess) {
        cudaGetLastError();
        return nullptr;
    }
    std::lock_guard<std::mutex> lock(g_mutex);
    CtrlState &c = g_ctrl_state[dev];
    if (!c.looked_up && cs == cudaStreamCaptureStatusActive) return nullptr;  // look it up outside a capture
    if (!c.looked_up) {
        c.looked_up = true;
        void *ptr = nullptr;
        if (cudaGetSymbolAddress(&ptr, g_ctrl) == cudaSuccess) {
            c.base = static_cast<unsigned *>(ptr);
        } else {
            cudaGetLastError();
        }
    }
    if (c.base == nullptr) return nullptr;
    int slot = -1;
    if (cs == cudaStreamCaptureStatusActive) {
        if (c.next_graph < kCtrlSlots) slot = c.next_graph++;
    } else {
        for (int i = 0; i < c.n_stream; ++i)
            if (c.stream_of[i] == sid) slot = i;
        if (slot < 0 && c.n_stream < kCtrlStreamSlots) {
            slot = c.n_stream++;
            c.stream_of[slot] = sid;
        }
    }
    return slot < 0 ? nullptr : c.base + static_cast<size_t>(slot) * kCtrlWords;
}

// Every launch of one call, given the plan and a workspace of p.ws_bytes.
// Where the one-launch path's group-barrier counters live: a self-clearing
// slot of the static table (or, when none is free, the workspace zeroed by a
// memset), or the head of a workspace that is zero when the call starts and
// that each launch leaves at zero (caller-owned and static workspaces).
enum CounterMode { kCountersSlot = 0, kCountersWorkspace = 1 };

int launch_all(const void *q, const void *k, const float *w, const void *mask, long long n_q, long long n_kv, int H,
               int D, int top_k, int32_t *out_idx, float *out_score, cudaStream_t st, int dtype,
               const lid_options *opt, const Plan &p, DeviceInfo &dev, uint8_t *ws,
               const int32_t *row_lo = nullptr, const int32_t *row_hi = nullptr, const float *q_scale = nullptr,
               const float *k_scale = nullptr, int counters = kCountersSlot) {
    if (n_kv == 0) {
        const long long n = n_q * top_k;
        long long blocks = (n + 255) / 256;
        if (blocks > 65535) blocks = 65535;
        fill_empty_kernel<<<static_cast<unsigned>(blocks), 256, 0, st>>>(out_idx, out_score, n);
        return cuda_status(cudaGetLastError());
    }
    CUtensorMap tmk, tmq;
    const int esize = dtype == LID_DTYPE_E4M3 ? 1 : 2;
    int rc = encode_2d(&tmk, k, static_cast<unsigned long long>(D), static_cast<unsigned long long>(n_kv), esize, kBM);
    if (!rc)
        rc = encode_2d(&tmq, q, static_cast<unsigned long long>(D), static_cast<unsigned long long>(n_q * H), esize,
                       static_cast<unsigned>(p.N));
    if (rc) return rc;
    ScoreParams sp = {};
    sp.mask = static_cast<const uint16_t *>(mask);
    sp.row_lo = row_lo;
    sp.row_hi = row_hi;
    sp.w = w;
    sp.q_scale = dtype == LID_DTYPE_E4M3 ? q_scale : nullptr;
    sp.k_scale = dtype == LID_DTYPE_E4M3 ? k_scale : nullptr;
    sp.esize = esize;
    sp.out_idx = out_idx;
    sp.out_score = out_score;
    sp.part = (!p.fused && p.splits > 1) ? reinterpret_cast<uint64_t *>(ws + kCounterBytes) : nullptr;
    sp.n_q = n_q;
    sp.n_kv = n_kv;
    sp.D = D;
    sp.QG = p.qg;
    sp.N = p.N;
    sp.top_k = top_k;
    sp.P = p.P;
    sp.n_groups = p.n_groups;
    sp.splits = p.splits;
    sp.tiles_per_split = p.tps;
    sp.n_tiles = p.n_tiles;
    sp.kstages = p.kstages;
    sp.acc_stages = p.acc_stages;
    sp.cap = p.cap;
    sp.tmem_cols = p.tmem_cols;
    sp.idesc = make_idesc(kBM, p.N, dtype == LID_DTYPE_BF16 ? 1 : 0);  // E4M3: format 0 of kind::f8f6f4
    sp.wait_limit = kWaitLimitCycles;
    sp.fault = 0;
    sp.tilepar = p.tilepar;
    if (p.single) {
        // the key-side data as bulk copies where their rows start 16-byte aligned
        sp.side_bulk = ((mask != nullptr && aligned(mask, 16) && (n_q == 1 || n_kv % 8 == 0)) ? 1 : 0) |
                       ((sp.k_scale != nullptr && aligned(sp.k_scale, 16)) ? 2 : 0);
        sp.f_count = reinterpret_cast<int *>(ws + p.off_count);
        sp.f_stats = reinterpret_cast<uint64_t *>(ws + p.off_stats);
        sp.f_reg = reinterpret_cast<uint64_t *>(ws + p.off_reg);
        sp.f_cand = reinterpret_cast<uint64_t *>(ws + p.off_cand);
        sp.f_cap = p.f_cap;
        sp.f_regcap = p.f_regcap;
        sp.f_pub = p.f_pub;
    }
    if (p.fused) {
        sp.f_bar = reinterpret_cast<unsigned *>(ws);
        sp.f_done = nullptr;
        if (!p.single) {
            sp.f_count = reinterpret_cast<int *>(ws + p.off_count);
            sp.f_hist = reinterpret_cast<int *>(ws + p.off_hist);
            sp.f_stats = reinterpret_cast<uint64_t *>(ws + p.off_stats);
            sp.f_cand = reinterpret_cast<uint64_t *>(ws + p.off_cand);
            sp.f_cap = p.f_cap;
            sp.f_early = p.early ? 1 : 0;
            sp.f_pub = p.f_pub;
            sp.f_reg = p.f_regcap > 0 ? reinterpret_cast<uint64_t *>(ws + p.off_reg) : nullptr;
            sp.f_regcap = p.f_regcap;
        }
        // the group barriers count arrivals from zero; everything else the
        // kernel reads it writes first
        if (counters == kCountersWorkspace) {
            sp.f_done = sp.f_bar + p.n_groups;  // zero on entry, left zero by the launch
        } else {
            unsigned *slot = ctrl_slot(st, p.n_groups);
            if (slot != nullptr) {
                sp.f_bar = slot;
                sp.f_done = slot + p.n_groups;
            } else {
                rc = cuda_status(cudaMemsetAsync(ws, 0, static_cast<size_t>(p.n_groups) * 4, st));
                if (rc) return rc;
            }
        }
    }
    if (opt && (opt->fault_inject == 2 || opt->fault_inject == 3)) {
        // test hooks: one wait that nothing completes, with a short limit
        sp.fault = opt->fault_inject;
        sp.wait_limit = 1ll << 22;
    }
    if (p.off_qbound > 0) {
        sp.qbound = reinterpret_cast<unsigned long long *>(ws + p.off_qbound);
        rc = cuda_status(cudaMemsetAsync(sp.qbound, 0, static_cast<size_t>(n_q) * 8, st));
        if (rc) return rc;
    }
    if (opt && opt->ev_score_begin) rc = record_event(opt->ev_score_begin, st);
    if (!rc) switch (H) {
        case 8: rc = launch_score_h<8>(tmk, tmq, sp, p, dev, 0, st); break;
        case 16: rc = launch_score_h<16>(tmk, tmq, sp, p, dev, 1, st); break;
        case 32: rc = launch_score_h<32>(tmk, tmq, sp, p, dev, 2, st); break;
        default: rc = launch_score_h<64>(tmk, tmq, sp, p, dev, 3, st); break;
    }
    if (!rc && opt && opt->ev_score_end) rc = record_event(opt->ev_score_end, st);
    if (rc || p.fused || p.splits == 1) return rc;
    // a few lists per query: the ranking merge (short CTAs, no shared-memory opt-in)
    const bool ranked = p.splits <= kRankMaxSplits && p.splits * top_k <= kRankMaxKeys;
    if (!ranked && !dev.attr_set[4]) {
        rc = cuda_status(cudaFuncSetAttribute(merge_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, dev.smem_optin));
        if (!rc)
            rc = cuda_status(cudaFuncSetAttribute(merge_kernel, cudaFuncAttributePreferredSharedMemoryCarveout,
                                                  cudaSharedmemCarveoutMaxShared));
        if (rc) return rc;
        dev.attr_set[4] = true;
    }
    MergeParams mp;
    mp.part = reinterpret_cast<const uint64_t *>(ws + kCounterBytes);
    mp.out_idx = out_idx;
    mp.out_score = out_score;
    mp.n_q = n_q;
    mp.splits = p.splits;
    mp.top_k = top_k;
    // programmatic dependent launch: the merge grid may be scheduled as the
    // scoring CTAs finish; it waits (griddepcontrol.wait) for their results
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(n_q));
    cfg.blockDim = dim3(ranked ? kRankThreads : kMergeThreads);
    cfg.dynamicSmemBytes = ranked ? static_cast<size_t>(p.splits) * top_k * 8 : p.merge_smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cuda_status(cudaLaunchKernelEx(&cfg, ranked ? merge_ranked_kernel : merge_kernel, mp));
}

int run(const void *q, const void *k, const float *w, const void *mask, long long n_q, long long n_kv, int H,
        int D, int top_k, int32_t *out_idx, float *out_score, void *stream, int dtype, const lid_options *opt,
        const int32_t *row_lo = nullptr, const int32_t *row_hi = nullptr, const float *q_scale = nullptr,
        const float *k_scale = nullptr) {
    DeviceInfo *dev = nullptr;
    Plan p;
    int rc = prepare(q, k, w, mask, n_q, n_kv, H, D, top_k, out_idx, out_score, dtype, opt, &dev, &p, row_lo, row_hi,
                     q_scale, k_scale);
    if (rc || n_q == 0) return rc;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    uint8_t *ws = nullptr;
    if (n_kv > 0 && p.ws_bytes > 0) {
        if (opt && opt->fault_inject == 1) return LID_ERR_OOM;
        if (ws_alloc(reinterpret_cast<void **>(&ws), static_cast<size_t>(p.ws_bytes), st, *dev) != cudaSuccess) {
            cudaGetLastError();
            return LID_ERR_OOM;
        }
    }
    rc = launch_all(q, k, w, mask, n_q, n_kv, H, D, top_k, out_idx, out_score, st, dtype, opt, p, *dev, ws, row_lo,
                    row_hi, q_scale, k_scale);
    if (ws) {
        const int frc = cuda_status(cudaFreeAsync(ws, st));
        if (!rc) rc = frc;
    }
    return rc;
}

// ------------------------------------------------------------------------
// No-allocation variant (lid_topk_static). Its split workspace lives in the
// fixed device array below instead of being allocated per call, for callers
// that cannot allocate device memory at call time.
constexpr size_t kStaticScratchBytes = 8u << 20;  // 8 MiB, held by every device that loads the library

static __device__ __align__(256) unsigned char g_lid_static_scratch[kStaticScratchBytes];

// Device address of the scratch array, looked up once per device and context
// (with that device current; g_static_scratch_ptr). In host code the array's
// name is only a stand-in for the symbol, never an address a kernel may use.
// The lookup is not a stream operation, so it is refused inside a capture.
int static_scratch(void **out, cudaStream_t st) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return LID_ERR_CUDA;
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(st, &cs) != cudaSuccess) return cuda_status(cudaGetLastError());
    std::lock_guard<std::mutex> lock(g_mutex);
    if (g_static_scratch_ptr[dev] == nullptr) {
        if (cs != cudaStreamCaptureStatusNone) return LID_ERR_INVALID_ARG;  // first call inside a capture
        void *ptr = nullptr;
        const int rc = cuda_status(cudaGetSymbolAddress(&ptr, g_lid_static_scratch));
        if (rc) return rc;
        g_static_scratch_ptr[dev] = ptr;
    }
    *out = g_static_scratch_ptr[dev];
    return LID_OK;
}

int run_static(const void *q, const void *k, const float *w, const void *mask, long long n_q, long long n_kv,
               int H, int D, int top_k, int32_t *out_idx, float *out_score, void *stream, int dtype) {
    DeviceInfo *dev = nullptr;
    Plan p;
    int rc = prepare(q, k, w, mask, n_q, n_kv, H, D, top_k, out_idx, out_score, dtype, nullptr, &dev, &p);
    if (rc || n_q == 0) return rc;
    if (static_cast<unsigned long long>(p.ws_bytes) > kStaticScratchBytes) return LID_ERR_SCRATCH_TOO_SMALL;
    uint8_t *ws = nullptr;
    if (n_kv > 0 && p.ws_bytes > 0) {
        void *scratch = nullptr;
        rc = static_scratch(&scratch, static_cast<cudaStream_t>(stream));
        if (rc) return rc;
        // the kernels write every entry they read, except the one-launch path's
        // barrier counters at the head, which are zero when the module loads and
        // which every launch leaves at zero
        ws = static_cast<uint8_t *>(scratch);
    }
    return launch_all(q, k, w, mask, n_q, n_kv, H, D, top_k, out_idx, out_score, static_cast<cudaStream_t>(stream),
                      dtype, nullptr, p, *dev, ws, nullptr, nullptr, nullptr, nullptr, kCountersWorkspace);
}

// Caller-owned workspace (lid_topk_ws): no allocation, no library state.
int run_ws(const void *q, const float *q_scale, const void *k, const float *k_scale, const float *w,
           const void *mask, const int32_t *row_lo, const int32_t *row_hi, long long n_q, long long n_kv, int H,
           int D, int top_k, int32_t *out_idx, float *out_score, void *workspace, long long ws_bytes, void *stream,
           int dtype, const lid_options *opt) {
    DeviceInfo *dev = nullptr;
    Plan p;
    if (opt && opt->fault_inject == 1) return LID_ERR_INVALID_ARG;  // (an allocation failure: nothing is allocated)
    int rc = prepare(q, k, w, mask, n_q, n_kv, H, D, top_k, out_idx, out_score, dtype, opt, &dev, &p, row_lo, row_hi,
                     q_scale, k_scale);
    if (rc || n_q == 0) return rc;
    uint8_t *ws = nullptr;
    if (n_kv > 0 && p.ws_bytes > 0) {
        if (workspace == nullptr || ws_bytes < p.ws_bytes) return LID_ERR_SCRATCH_TOO_SMALL;
        if (!aligned(workspace, 256)) return LID_ERR_INVALID_ARG;
        ws = static_cast<uint8_t *>(workspace);
    }
    return launch_all(q, k, w, mask, n_q, n_kv, H, D, top_k, out_idx, out_score, static_cast<cudaStream_t>(stream),
                      dtype, opt, p, *dev, ws, row_lo, row_hi, q_scale, k_scale, kCountersWorkspace);
}

}  // namespace

// ---- shared with the sparse-attention translation unit (lid_internal.h)
int env_device(DeviceEnv *env) {
    DeviceInfo *dev = nullptr;
    if (device_info(&dev)) return LID_ERR_CUDA;
    env->sm103 = dev->sm103;
    env->sm_count = dev->sm_count;
    env->smem_optin = dev->smem_optin;
    env->ctx_id = dev->ctx_id;
    return LID_OK;
}

int env_cuda_status(cudaError_t e) { return cuda_status(e); }

cudaError_t env_ws_alloc(void **ptr, size_t bytes, cudaStream_t st) {
    DeviceInfo *dev = nullptr;
    if (device_info(&dev)) return cudaErrorInvalidDevice;
    return ws_alloc(ptr, bytes, st, *dev);
}

}  // namespace lid

extern "C" {

int lid_topk(const void *q, const void *k, const float *w, const void *mask, int64_t n_q, int64_t n_kv, int H,
             int D, int top_k, int32_t *out_idx, float *out_score, void *stream) {
    return lid::run(q, k, w, mask, n_q, n_kv, H, D, top_k, out_idx, out_score, stream, LID_DTYPE_BF16, nullptr);
}

int lid_topk_f16(const void *q, const void *k, const float *w, const void *mask, int64_t n_q, int64_t n_kv, int H,
                 int D, int top_k, int32_t *out_idx, float *out_score, void *stream) {
    return lid::run(q, k, w, mask, n_q, n_kv, H, D, top_k, out_idx, out_score, stream, LID_DTYPE_F16, nullptr);
}

int lid_topk_ex(const void *q, const void *k, const float *w, const void *mask, int64_t n_q, int64_t n_kv, int H,
                int D, int top_k, int32_t *out_idx, float *out_score, void *stream, int dtype,
                const lid_options *opt) {
    if (dtype == LID_DTYPE_E4M3) return LID_ERR_INVALID_ARG;  // 8-bit operands come with scales: lid_topk_e4m3
    return lid::run(q, k, w, mask, n_q, n_kv, H, D, top_k, out_idx, out_score, stream, dtype, opt);
}

int lid_topk_ranges(const void *q, const void *k, const float *w, const int32_t *row_lo, const int32_t *row_hi,
                    int64_t n_q, int64_t n_kv, int H, int D, int top_k, int32_t *out_idx, float *out_score,
                    void *stream, int dtype, const lid_options *opt) {
    if (n_q > 0 && (row_lo == nullptr || row_hi == nullptr)) return LID_ERR_INVALID_ARG;
    if (dtype == LID_DTYPE_E4M3) return LID_ERR_INVALID_ARG;
    return lid::run(q, k, w, nullptr, n_q, n_kv, H, D, top_k, out_idx, out_score, stream, dtype, opt, row_lo, row_hi);
}

int lid_topk_e4m3(const void *q8, const float *q_scale, const void *k8, const float *k_scale, const float *w,
                  const void *mask, const int32_t *row_lo, const int32_t *row_hi, int64_t n_q, int64_t n_kv, int H,
                  int D, int top_k, int32_t *out_idx, float *out_score, void *stream, const lid_options *opt) {
    return lid::run(q8, k8, w, mask, n_q, n_kv, H, D, top_k, out_idx, out_score, stream, LID_DTYPE_E4M3, opt, row_lo,
                    row_hi, q_scale, k_scale);
}

namespace {

// The copy stream and events of the host-buffer calls on this device, made on
// first use (called with g_host_mutex held).
bool host_copy_state(lid::DeviceInfo &d) {
    if (d.copy_stream != nullptr) return true;
    cudaStream_t cs = nullptr;
    if (cudaStreamCreateWithFlags(&cs, cudaStreamNonBlocking) != cudaSuccess) {
        cudaGetLastError();
        return false;
    }
    for (int i = 0; i < 2; ++i) {
        if (cudaEventCreateWithFlags(&d.host_copied[i], cudaEventDisableTiming) != cudaSuccess ||
            cudaEventCreateWithFlags(&d.host_done[i], cudaEventDisableTiming) != cudaSuccess) {
            cudaGetLastError();
            return false;  // the stream stays unset: the next call tries again
        }
    }
    d.copy_stream = cs;
    return true;
}

// The host-buffer call up to its last enqueued copy; *enqueued tells whether
// anything reached the stream (argument errors return before that).
//
// The input copies run on the device's copy stream, which does not wait for
// earlier work on `stream`; the kernels, the result copies and the release of
// the staging run on `stream` after them. So calls on one stream overlap one
// call's input copies with the previous call's kernels, while the kernels
// themselves run one after another. A call's copies wait for the end of the
// call two before it (on whatever stream), which bounds the staging alive at
// once to three calls. Inside a stream capture everything stays on `stream`.
int topk_host_enqueue(const void *q, const void *k, const float *w, const void *mask, int64_t n_q, int64_t n_kv, int H,
                      int D, int top_k, int32_t *out_idx, float *out_score, void *stream, int dtype, bool *enqueued) {
    *enqueued = false;
    int rc = lid::validate_shape(n_q, n_kv, H, D, top_k);
    if (rc) return rc;
    if (dtype != LID_DTYPE_BF16 && dtype != LID_DTYPE_F16) return LID_ERR_INVALID_ARG;
    if (n_q == 0) return LID_OK;
    if (!out_idx || !out_score || (n_kv > 0 && (!q || !k || !w))) return LID_ERR_INVALID_ARG;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const size_t qb = static_cast<size_t>(n_q) * H * D * 2, kb = static_cast<size_t>(n_kv) * D * 2;
    const size_t wb = static_cast<size_t>(n_q) * H * 4, mb = mask ? static_cast<size_t>(n_q) * n_kv * 2 : 0;
    const size_t ob = static_cast<size_t>(n_q) * top_k * 4;
    auto up = [](size_t x) { return (x + 255) & ~static_cast<size_t>(255); };
    const size_t total = up(qb) + up(kb) + up(wb) + up(mb) + 2 * up(ob);
    lid::DeviceInfo *dev = nullptr;
    rc = lid::device_info(&dev);
    if (rc) return rc;
    cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(st, &cap) != cudaSuccess) {
        cudaGetLastError();
        return LID_ERR_CUDA;
    }
    std::lock_guard<std::mutex> lock(lid::g_host_mutex);
    const bool split = cap == cudaStreamCaptureStatusNone && host_copy_state(*dev);
    cudaStream_t cs = split ? dev->copy_stream : st;
    const int slot = static_cast<int>(dev->host_calls & 1ull);
    if (split && dev->host_calls >= 2 && cudaStreamWaitEvent(cs, dev->host_done[slot], 0) != cudaSuccess)
        return lid::cuda_status(cudaGetLastError());
    uint8_t *d = nullptr;
    if (lid::ws_alloc(reinterpret_cast<void **>(&d), total, cs, *dev) != cudaSuccess) {
        cudaGetLastError();
        return LID_ERR_OOM;
    }
    *enqueued = true;
    uint8_t *dq = d, *dk = dq + up(qb), *dw = dk + up(kb), *dm = dw + up(wb), *di = dm + up(mb), *ds = di + up(ob);
    bool ok = true;
    if (qb) ok = ok && cudaMemcpyAsync(dq, q, qb, cudaMemcpyHostToDevice, cs) == cudaSuccess;
    if (kb) ok = ok && cudaMemcpyAsync(dk, k, kb, cudaMemcpyHostToDevice, cs) == cudaSuccess;
    if (wb) ok = ok && cudaMemcpyAsync(dw, w, wb, cudaMemcpyHostToDevice, cs) == cudaSuccess;
    if (mb) ok = ok && cudaMemcpyAsync(dm, mask, mb, cudaMemcpyHostToDevice, cs) == cudaSuccess;
    // `stream` takes over after the copies (also when one failed to enqueue, so
    // that the staging is released after whatever was enqueued)
    bool joined = !split;
    if (split) {
        joined = cudaEventRecord(dev->host_copied[slot], cs) == cudaSuccess &&
                 cudaStreamWaitEvent(st, dev->host_copied[slot], 0) == cudaSuccess;
        if (!joined) cudaStreamSynchronize(cs);  // the copies are done before the staging is released on `stream`
    }
    // a failed enqueue is an error even if the runtime no longer reports it
    auto enqueue_error = []() {
        const cudaError_t e = cudaGetLastError();
        return e != cudaSuccess ? lid::cuda_status(e) : LID_ERR_CUDA;
    };
    rc = ok && joined ? lid::run(dq, dk, reinterpret_cast<const float *>(dw), mask ? dm : nullptr, n_q, n_kv, H, D,
                                 top_k, reinterpret_cast<int32_t *>(di), reinterpret_cast<float *>(ds), stream, dtype,
                                 nullptr)
                      : enqueue_error();
    if (!rc) {
        ok = cudaMemcpyAsync(out_idx, di, ob, cudaMemcpyDeviceToHost, st) == cudaSuccess &&
             cudaMemcpyAsync(out_score, ds, ob, cudaMemcpyDeviceToHost, st) == cudaSuccess;
        if (!ok) rc = enqueue_error();
    }
    cudaFreeAsync(d, st);
    if (split) {
        if (cudaEventRecord(dev->host_done[slot], st) == cudaSuccess) {
            ++dev->host_calls;
        } else {
            cudaGetLastError();
            cudaStreamSynchronize(st);  // the slot's event is stale: make the bound hold by waiting here
            ++dev->host_calls;
        }
    }
    return rc;
}

}  // namespace

int lid_topk_host(const void *q, const void *k, const float *w, const void *mask, int64_t n_q, int64_t n_kv, int H,
                  int D, int top_k, int32_t *out_idx, float *out_score, void *stream, int dtype) {
    // Once anything is enqueued the stream is drained, errors included, so that
    // no copy from or to the caller's host buffers is in flight when this returns.
    bool enqueued = false;
    const int rc = topk_host_enqueue(q, k, w, mask, n_q, n_kv, H, D, top_k, out_idx, out_score, stream, dtype,
                                     &enqueued);
    const bool drained = !enqueued || cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) == cudaSuccess;
    return rc ? rc : drained ? LID_OK : LID_ERR_CUDA;
}

int lid_topk_host_async(const void *q, const void *k, const float *w, const void *mask, int64_t n_q, int64_t n_kv,
                        int H, int D, int top_k, int32_t *out_idx, float *out_score, void *stream, int dtype) {
    bool enqueued = false;
    return topk_host_enqueue(q, k, w, mask, n_q, n_kv, H, D, top_k, out_idx, out_score, stream, dtype, &enqueued);
}

int lid_plan(int64_t n_q, int64_t n_kv, int H, int D, int top_k, const lid_options *opt, lid_plan_info *info) {
    if (!info) return LID_ERR_INVALID_ARG;
    int rc = lid::validate_shape(n_q, n_kv, H, D, top_k);
    if (rc) return rc;
    lid::DeviceInfo *dev = nullptr;
    rc = lid::device_info(&dev);
    if (rc) return rc;
    lid::Plan p;
    rc = lid::make_plan(n_q, n_kv, H, D, top_k, opt, *dev, &p, opt != nullptr && opt->plan_ranges != 0);
    if (rc) return rc;
    info->qg = p.qg;
    info->n_groups = p.n_groups;
    info->splits = p.splits;
    info->tiles_per_split = p.tps;
    info->kstages = p.kstages;
    info->acc_stages = p.acc_stages;
    info->cap = p.cap;
    info->threads = p.threads;
    info->smem_bytes = static_cast<int>(p.smem);
    info->fused = p.single ? 2 : (p.fused ? 1 : 0);
    info->workspace_bytes = p.ws_bytes;
    return LID_OK;
}

int lid_device_error(int reset) {
    if (cudaDeviceSynchronize() != cudaSuccess) return -1;
    int v = 0;
    if (cudaMemcpyFromSymbol(&v, lid::g_dev_error, sizeof(int)) != cudaSuccess) return -1;
    if (reset) {
        const int z = 0;
        if (cudaMemcpyToSymbol(lid::g_dev_error, &z, sizeof(int)) != cudaSuccess) return -1;
    }
    const int va = lid::attn_device_error(reset);  // the sparse-attention kernels' word
    if (va < 0) return -1;
    return v ? v : va;
}

int lid_topk_ws(const void *q, const float *q_scale, const void *k, const float *k_scale, const float *w,
                const void *mask, const int32_t *row_lo, const int32_t *row_hi, int64_t n_q, int64_t n_kv, int H, int D,
                int top_k, int32_t *out_idx, float *out_score, void *workspace, int64_t workspace_bytes, void *stream,
                int dtype, const lid_options *opt) {
    if (n_q > 0 && (row_lo == nullptr) != (row_hi == nullptr)) return LID_ERR_INVALID_ARG;
    return lid::run_ws(q, dtype == LID_DTYPE_E4M3 ? q_scale : nullptr, k, dtype == LID_DTYPE_E4M3 ? k_scale : nullptr,
                       w, mask, row_lo, row_hi, n_q, n_kv, H, D, top_k, out_idx, out_score, workspace, workspace_bytes,
                       stream, dtype, opt);
}

int lid_topk_static(const void *q, const void *k, const float *w, const void *mask, int64_t n_q, int64_t n_kv,
                    int H, int D, int top_k, int32_t *out_idx, float *out_score, void *stream, int dtype) {
    if (dtype == LID_DTYPE_E4M3) return LID_ERR_INVALID_ARG;
    return lid::run_static(q, k, w, mask, n_q, n_kv, H, D, top_k, out_idx, out_score, stream, dtype);
}

const char *lid_last_cuda_error(void) {
    return lid::g_last_cuda_error == cudaSuccess ? "no error" : cudaGetErrorString(lid::g_last_cuda_error);
}

const char *lid_status_string(int status) {
    switch (status) {
        case LID_OK: return "ok";
        case LID_ERR_INVALID_ARG: return "invalid argument (null or misaligned pointer, negative size)";
        case LID_ERR_UNSUPPORTED: return "unsupported shape or device (H, D, top_k, sizes, or not sm_103)";
        case LID_ERR_OOM: return "workspace allocation failed";
        case LID_ERR_CUDA: return "CUDA runtime error";
        case LID_ERR_DEVICE_TIMEOUT: return "a bounded device-side wait ran out";
        case LID_ERR_SCRATCH_TOO_SMALL:
            return "the shape needs more split workspace than the given (or lid_topk_static's fixed 8 MiB) scratch";
        default: return "unknown status";
    }
}

}  // extern "C"
