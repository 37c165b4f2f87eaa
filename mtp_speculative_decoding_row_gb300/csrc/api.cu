// api.cu -- the C ABI (include/mtp_rs.h): argument validation, launch
// planning (cluster size, shared memory) and cluster launches.
#include <cuda_runtime.h>

#include <cstdint>
#include <cstdlib>
#include <mutex>
#include <vector>

#include "common.cuh"
#include "kernels.h"
#include "mtp_rs.h"

namespace {

using namespace mtp;

constexpr uint32_t kMaxSmem = 232448;        // 227 KB per CTA on sm_100-class parts
constexpr uint32_t kRowBudget = 100 * 1024;  // row kernel: two CTAs per SM
constexpr uint32_t kTVBudget = 110 * 1024;   // TV kernel: two CTAs per SM

struct Plan {
    int C = 0;
    uint32_t slice_bytes = 0;
    uint32_t smem = 0;
    int nres = 0;
};

struct CacheEntry {
    int device;
    const void *func;
    int C;
    uint32_t smem;
    int ok;
};

std::mutex g_mu;
std::vector<CacheEntry> g_cache;
std::vector<std::pair<int, const void *>> g_attr_done;

int env_cluster() {
    const char *e = std::getenv("MTP_RS_CLUSTER");
    if (!e) return 0;
    const int c = std::atoi(e);
    return (c == 1 || c == 2 || c == 4 || c == 8 || c == 16) ? c : 0;
}

int env_int(const char *name) {
    const char *e = std::getenv(name);
    return e ? std::atoi(e) : 0;
}

// Set the function attributes once per device and kernel.
cudaError_t prepare_func(int dev, const void *func) {
    std::lock_guard<std::mutex> lk(g_mu);
    for (auto &p : g_attr_done)
        if (p.first == dev && p.second == func) return cudaSuccess;
    int optin = 0;
    cudaError_t e = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(optin < static_cast<int>(kMaxSmem) ? optin : kMaxSmem));
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(func, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (e != cudaSuccess) return e;
    g_attr_done.emplace_back(dev, func);
    return cudaSuccess;
}

// Whether clusters of C CTAs with `smem` bytes each can be resident.
bool cluster_fits(int dev, const void *func, int C, uint32_t smem) {
    {
        std::lock_guard<std::mutex> lk(g_mu);
        for (auto &c : g_cache)
            if (c.device == dev && c.func == func && c.C == C && c.smem == smem) return c.ok != 0;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(C);
    cfg.blockDim = dim3(NT);
    cfg.dynamicSmemBytes = smem;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = C;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    const cudaError_t e = cudaOccupancyMaxActiveClusters(&n, func, &cfg);
    const int ok = (e == cudaSuccess && n > 0) ? 1 : 0;
    if (e != cudaSuccess) (void)cudaGetLastError();
    std::lock_guard<std::mutex> lk(g_mu);
    g_cache.push_back({dev, func, C, smem, ok});
    return ok != 0;
}

// Row kernel: two row slices per CTA.  Smallest cluster under the budget.
bool plan_row(int dev, const void *func, int V, int es, Plan &p) {
    const int forced = env_cluster();
    for (int C = 1; C <= MAX_C; C *= 2) {
        if (forced && C != forced) continue;
        const uint32_t sb = slice_buffer_bytes(V, es, C);
        const uint32_t smem = HDR_BYTES + 2 * sb;
        if (smem > kMaxSmem) continue;
        if (!forced && smem > kRowBudget && C < MAX_C) continue;
        if (!cluster_fits(dev, func, C, smem)) continue;
        p = {C, sb, smem, 0};
        return true;
    }
    return false;
}

// TV kernel: one target slice, nres draft slices and gamma bit rows.
bool plan_tv(int dev, const void *func, int V, int es, int gamma, Plan &p) {
    const int forced = env_cluster();
    for (int pass = 0; pass < 2; ++pass) {
        for (int C = 1; C <= MAX_C; C *= 2) {
            if (forced && C != forced) continue;
            const uint32_t sb = slice_buffer_bytes(V, es, C);
            const uint32_t bitb = static_cast<uint32_t>(gamma) * static_cast<uint32_t>(slice_vectors(V, 16 / es, C));
            const uint32_t fixed = HDR_BYTES + sb + ((bitb + 127u) & ~127u);
            const uint32_t budget = (pass == 0 && !forced) ? kTVBudget : kMaxSmem;
            if (fixed + sb > budget) continue;
            int nres = static_cast<int>((budget - fixed) / sb);
            if (nres > gamma) nres = gamma;
            const int cap = env_int("MTP_RS_TV_NRES");
            if (cap > 0 && nres > cap) nres = cap;
            if (pass == 0 && !forced && nres < gamma && C < MAX_C) continue;
            const uint32_t smem = fixed + static_cast<uint32_t>(nres) * sb;
            if (!cluster_fits(dev, func, C, smem)) continue;
            p = {C, sb, smem, nres};
            return true;
        }
    }
    return false;
}

int launch(const void *func, const Plan &p, int units, void *args, mtp_stream_t stream) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(units) * static_cast<unsigned>(p.C));
    cfg.blockDim = dim3(NT);
    cfg.dynamicSmemBytes = p.smem;
    cfg.stream = reinterpret_cast<cudaStream_t>(stream);
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = p.C;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    void *kargs[] = {args};
    const cudaError_t e = cudaLaunchKernelExC(&cfg, func, kargs);
    return e == cudaSuccess ? MTP_OK : MTP_ERR_CUDA;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int esize(mtp_dtype d) { return d == MTP_DTYPE_F32 ? 4 : 2; }

int current_device(int &dev) {
    if (cudaGetDevice(&dev) != cudaSuccess) {
        (void)cudaGetLastError();
        return MTP_ERR_CUDA;
    }
    return MTP_OK;
}

int row_call(int mode, const void *target, const void *draft, mtp_dtype dtype, const int32_t *ids,
             const float *temp, const float *unif, int B, int gamma, int V, int32_t *tokens, int32_t *accept_len,
             float *alpha, float *entropy, int32_t *flags, mtp_stream_t stream) {
    if (dtype != MTP_DTYPE_F32 && dtype != MTP_DTYPE_BF16) return MTP_ERR_UNSUPPORTED_DTYPE;
    if (B < 0 || gamma < 1 || gamma > MTP_MAX_GAMMA || V < 1) return MTP_ERR_INVALID_ARG;
    if (B == 0) return MTP_OK;
    if (!target || !draft || !temp) return MTP_ERR_INVALID_ARG;
    if (!aligned16(target) || !aligned16(draft)) return MTP_ERR_MISALIGNED;
    int dev;
    if (current_device(dev) != MTP_OK) return MTP_ERR_CUDA;
    const void *func = row_kernel(dtype == MTP_DTYPE_F32 ? 0 : 1, mode);
    if (prepare_func(dev, func) != cudaSuccess) return MTP_ERR_CUDA;
    const int es = esize(dtype);
    Plan p;
    if (!plan_row(dev, func, V, es, p)) return MTP_ERR_NO_DEVICE;
    VerifyArgs A;
    A.target = target;
    A.draft = draft;
    A.ids = ids;
    A.temp = temp;
    A.unif = unif;
    A.B = B;
    A.gamma = gamma;
    A.V = V;
    A.aligned = (V % (16 / es) == 0) ? 1 : 0;
    A.slice_bytes = p.slice_bytes;
    A.tokens = tokens;
    A.accept_len = accept_len;
    A.alpha = alpha;
    A.entropy = entropy;
    A.flags = flags;
    return launch(func, p, B, &A, stream);
}

}  // namespace

extern "C" int mtp_rs_verify(const void *target_logits, const void *draft_logits, mtp_dtype dtype,
                             const int32_t *draft_ids, const float *temperature, const float *uniforms, int B,
                             int gamma, int V, int32_t *out_tokens, int32_t *accept_len, float *alpha,
                             float *entropy, int32_t *row_flags, mtp_stream_t stream) {
    if (B > 0 && (!draft_ids || !uniforms || !out_tokens || !accept_len)) return MTP_ERR_INVALID_ARG;
    if ((alpha == nullptr) != (entropy == nullptr)) return MTP_ERR_INVALID_ARG;
    const int mode = alpha ? MODE_VERIFY_STATS : MODE_VERIFY;
    return row_call(mode, target_logits, draft_logits, dtype, draft_ids, temperature, uniforms, B, gamma, V,
                    out_tokens, accept_len, alpha, entropy, row_flags, stream);
}

extern "C" int mtp_row_stats(const void *target_logits, const void *draft_logits, mtp_dtype dtype,
                             const float *temperature, int B, int gamma, int V, float *alpha, float *entropy,
                             int32_t *row_flags, mtp_stream_t stream) {
    if (B > 0 && (!alpha || !entropy)) return MTP_ERR_INVALID_ARG;
    return row_call(MODE_STATS, target_logits, draft_logits, dtype, nullptr, temperature, nullptr, B, gamma, V,
                    nullptr, nullptr, alpha, entropy, row_flags, stream);
}

extern "C" int mtp_tv_loss_fwd_bwd(const void *target_logits, const void *draft_logits, mtp_dtype dtype,
                                   float temperature, int N, int gamma, int V, float grad_scale, float *loss,
                                   float *alpha, float *grad_draft_logits, int32_t *row_flags,
                                   mtp_stream_t stream) {
    if (dtype != MTP_DTYPE_F32 && dtype != MTP_DTYPE_BF16) return MTP_ERR_UNSUPPORTED_DTYPE;
    if (N < 0 || gamma < 1 || gamma > MTP_MAX_GAMMA || V < 1) return MTP_ERR_INVALID_ARG;
    if (N == 0) return MTP_OK;
    if (!target_logits || !draft_logits || !loss || !grad_draft_logits) return MTP_ERR_INVALID_ARG;
    if (!aligned16(target_logits) || !aligned16(draft_logits) || !aligned16(grad_draft_logits))
        return MTP_ERR_MISALIGNED;
    int dev;
    if (current_device(dev) != MTP_OK) return MTP_ERR_CUDA;
    const void *func = tv_kernel(dtype == MTP_DTYPE_F32 ? 0 : 1);
    if (prepare_func(dev, func) != cudaSuccess) return MTP_ERR_CUDA;
    const int es = esize(dtype);
    Plan p;
    if (!plan_tv(dev, func, V, es, gamma, p)) return MTP_ERR_NO_DEVICE;
    TVArgs A;
    A.target = target_logits;
    A.draft = draft_logits;
    A.temperature = temperature;
    A.grad_scale = grad_scale;
    A.N = N;
    A.gamma = gamma;
    A.V = V;
    A.aligned = (V % (16 / es) == 0) ? 1 : 0;
    A.nres = p.nres;
    A.slice_bytes = p.slice_bytes;
    A.loss = loss;
    A.alpha = alpha;
    A.grad = grad_draft_logits;
    A.flags = row_flags;
    return launch(func, p, N, &A, stream);
}

extern "C" const char *mtp_status_string(int status) {
    switch (status) {
        case MTP_OK: return "ok";
        case MTP_ERR_INVALID_ARG: return "invalid argument";
        case MTP_ERR_UNSUPPORTED_DTYPE: return "unsupported dtype";
        case MTP_ERR_MISALIGNED: return "logit or gradient base pointer not 16-byte aligned";
        case MTP_ERR_CUDA: return "CUDA error";
        case MTP_ERR_NO_DEVICE: return "no usable cluster launch configuration on this device";
        default: return "unknown status";
    }
}
