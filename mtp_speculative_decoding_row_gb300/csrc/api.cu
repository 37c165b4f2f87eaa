// api.cu -- the C ABI (include/mtp_rs.h): argument validation, launch
// planning (cluster size, shared memory) and cluster launches.
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>
#include <vector>

#include "common.cuh"
#include "kernels.h"
#include "gsample.h"
#include "mtp_rs.h"

namespace {

using namespace mtp;

constexpr uint32_t kMaxSmem = 232448;        // 227 KB per CTA on sm_100-class parts

struct Plan {
    int C = 0;
    uint32_t slice_bytes = 0;
    uint32_t smem = 0;
    int nres = 0;
    int clusters = 0;  // persistent grid: co-resident clusters used
    int streams = 1;   // row kernel: sequences in flight per CTA
    int threads = 0;   // threads per CTA
    int ring = 0;      // streaming kernel: chunk slots per warp
    int depth = 0;     // streaming kernel: look-ahead positions
    int cv = 0;        // streaming kernel: vectors of each row per chunk
    const void *func = nullptr;
    int seg_vectors = 0;
    bool pdl = false;  // the kernel waits for earlier launches itself (griddepcontrol): launch it programmatically
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

// Process-wide tuning overrides (mtp_set_tuning); all zero = the planners'
// own choices.  Read under the lock, once per call.
mtp_tuning g_tune = {};

mtp_tuning tuning() {
    std::lock_guard<std::mutex> lk(g_mu);
    return g_tune;
}

int tuned_cluster(const mtp_tuning &t) {
    const int c = t.cluster_size;
    return (c == 1 || c == 2 || c == 4 || c == 8 || c == 16) ? c : 0;
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

// Largest number of co-resident clusters of C CTAs with `smem` bytes each
// (0 when the configuration cannot run).
int max_clusters(int dev, const void *func, int C, uint32_t smem, int threads) {
    {
        std::lock_guard<std::mutex> lk(g_mu);
        for (auto &c : g_cache)
            if (c.device == dev && c.func == func && c.C == C && c.smem == smem) return c.ok;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(C);
    cfg.blockDim = dim3(threads);
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
    if (e != cudaSuccess) {
        (void)cudaGetLastError();
        n = 0;
    }
    std::lock_guard<std::mutex> lk(g_mu);
    g_cache.push_back({dev, func, C, smem, n});
    return n;
}

uint32_t smem_optin(int dev) {
    int optin = 0;
    if (cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess) {
        (void)cudaGetLastError();
        return 0;
    }
    return static_cast<uint32_t>(optin < static_cast<int>(kMaxSmem) ? optin : kMaxSmem);
}

// Persistent row kernel: `streams` (1 or 2) sequences in flight per CTA, one
// row pair slice each.  Picks the cluster size (1..16) and stream count that
// keep the most sequence slices in flight for `units` sequences; the grid is
// the co-resident cluster count.
bool plan_row(int dev, const void *func, int V, int es, int units, Plan &p) {
    const mtp_tuning tu = tuning();
    const int forced = tu.cluster_size;
    const int forced_ns = tu.row_streams;
    const uint32_t cap = smem_optin(dev);
    long best = -1;
    for (int ns = 1; ns <= 2; ++ns) {
        if (forced_ns && ns != forced_ns) continue;
        for (int C = 1; C <= MAX_C; ++C) {
            if (forced && C != forced) continue;
            const uint32_t sb = slice_buffer_bytes(V, es, C);
            const uint32_t smem = row_hdr_bytes() + 2 * ns * sb;
            if (smem > cap) continue;
            const int nc = max_clusters(dev, func, C, smem, row_threads());
            if (nc <= 0) continue;
            int used = nc < units ? nc : units;
            if (tu.max_clusters > 0 && used > tu.max_clusters) used = tu.max_clusters;
            const long inflight = static_cast<long>(nc) * ns < units ? static_cast<long>(nc) * ns : units;
            const long score = inflight * C * 4 + used;  // slices in flight, then clusters used
            if (score > best) {
                best = score;
                p = {C, sb, smem, 0, used, ns, row_threads()};
            }
        }
    }
    return best > 0;
}

// Streaming verify kernel: clusters of C CTAs x NT/32 warps, one vocabulary
// segment per warp, one sequence per cluster at a time.  Picks the cluster
// size with the smallest estimated makespan, ceil(units / clusters) waves of
// (1 / C + a fixed latency share) sequence-times, among sizes whose segments
// hold at least 64 vectors (or C = 1) and at most the chunk-list limit; ties
// go to more busy CTAs.
bool stream_usable(int V, int es, int gamma) {
    if (tuning().verify_kernel == MTP_KERNEL_RESIDENT) return false;
    return gamma <= stream_max_gamma() && V % (16 / es) == 0;
}

// Chunk size for a warp segment of nvs vectors: 3 KB chunks when the
// segment holds at least eight of them (fewer copies and less per-chunk
// control for the same bytes), else 2 KB chunks (less waste in the ragged
// last chunk of short segments).  The rejection-sampling verify kernel
// (mode 0), the streaming TV kernel (mode 3) and the row-pair kernel (mode
// 4) take 2.5 KB chunks: measured on GB300 they beat both at the B = 64 and
// B = 512 verify batches, the N = 16,384 TV batches and the B = 256
// diagnostics (fewer chunks than 2 KB, four CTAs per SM still fit, unlike
// 3 KB).
int stream_chunk_for(int nvs, int mode = -1) {
    const int forced = tuning().chunk_vectors;
    if (forced == 128 || forced == 192) return forced;
    if (forced == 160 && (mode == 0 || mode == 3 || mode == 4)) return forced;
    if (mode == 0 || mode == 3 || mode == 4) return 160;
    return nvs >= 8 * 192 ? 192 : 128;
}

bool plan_stream(int dev, int dtype, int V, int es, int gamma, int units, Plan &p, int mode = 0,
                 bool dbl = false) {
    const mtp_tuning tu = tuning();
    const int forced = tuned_cluster(tu);
    int R = tu.ring_slots;
    if (R < 2 || R > stream_max_ring()) R = 2;
    int depth = gamma;  // stream every position without waiting for decisions
    if (tu.lookahead > 0) depth = tu.lookahead - 1;
    if (depth < 0) depth = 0;
    if (depth > gamma) depth = gamma;
    const uint32_t cap = smem_optin(dev);
    const int nw = stream_threads() / 32;
    const int nv = V / (16 / es);
    double best = 1e30;
    long best_busy = -1;
    bool found = false;
    for (int C = 1; C <= MAX_C; ++C) {
        if (forced && C != forced) continue;
        const int S = C * nw;
        if (S > stream_max_segments()) continue;
        const int nvs = (nv + S - 1) / S;
        const int cv = mode == 1 ? 128 : stream_chunk_for(nvs, mode);
        if ((nvs + cv - 1) / cv > stream_max_chunks()) continue;
        if (!forced && C > 1 && nvs < 64) continue;
        const uint32_t smem = stream_hdr_bytes() + stream_rec_bytes(gamma, S) +
                              static_cast<uint32_t>(nw * R) * stream_slot_bytes(cv);
        if (smem > cap) continue;
        const void *func = stream_kernel(dtype, cv, mode, dbl && gamma == 0);
        if (prepare_func(dev, func) != cudaSuccess) return false;
        const int nc = max_clusters(dev, func, C, smem, stream_threads());
        if (nc <= 0) continue;
        int used = nc < units ? nc : units;
        if (tu.max_clusters > 0 && used > tu.max_clusters) used = tu.max_clusters;
        // per wave: the sequence's share of the row (1 / C) plus a fixed
        // latency term (exchanges, decision, sampling)
        const double est = static_cast<double>((units + used - 1) / used) * (1.0 / C + 0.03);
        const long busy = static_cast<long>(used) * C;
        if (est < best - 1e-12 || (est < best + 1e-12 && busy > best_busy)) {
            best = est;
            best_busy = busy;
            p = Plan{};
            p.C = C;
            p.smem = smem;
            p.clusters = used;
            p.threads = stream_threads();
            p.ring = R;
            p.depth = depth;
            p.seg_vectors = nvs;
            p.cv = cv;
            p.func = func;
            p.pdl = true;
            found = true;
        }
    }
    return found;
}

// Gumbel-max draft sampling (one pass per row): clusters of C CTAs, one row
// per cluster at a time.  Same estimate as plan_stream: waves of rows times
// each row's share (1 / C) plus a fixed term for the cluster barrier and the
// selection; rows too short for a cluster stay on one CTA.
bool plan_gsample(int dev, int dtype, int V, int es, int units, Plan &p) {
    const mtp_tuning tu = tuning();
    const int forced = tuned_cluster(tu);
    const void *func = gsample_kernel(dtype);
    if (prepare_func(dev, func) != cudaSuccess) return false;
    const int nw = gsample_threads() / 32;
    const int nv = V / (16 / es);
    const uint32_t smem = gsample_smem_bytes();
    double best = 1e30;
    bool found = false;
    for (int C = 1; C <= gsample_max_cluster(); ++C) {
        if (forced && C != forced) continue;
        if (!forced && C > 1 && (nv + C * nw - 1) / (C * nw) < 64) continue;
        const int nc = max_clusters(dev, func, C, smem, gsample_threads());
        if (nc <= 0) continue;
        int used = nc < units ? nc : units;
        if (tu.max_clusters > 0 && used > tu.max_clusters) used = tu.max_clusters;
        const double est = static_cast<double>((units + used - 1) / used) * (1.0 / C + 0.03);
        if (est < best - 1e-12) {
            best = est;
            p = Plan{};
            p.C = C;
            p.smem = smem;
            p.clusters = used;
            p.threads = gsample_threads();
            p.func = func;
            found = true;
        }
    }
    return found;
}

// Streaming TV kernel: clusters of C CTAs x NT/32 warps, one vocabulary
// segment per warp, one position per cluster at a time.  Among cluster sizes
// (powers of two) whose shared memory fits, the one with the most warps in
// flight wins; within 5 % the larger cluster (shorter per-position chain).  Measured on
// GB300, concurrency matters more than keeping every re-read row in L2, so
// the positions in flight are capped only when mtp_tuning.tv_l2_mb sets an L2
// budget for the 2 gamma rows a position re-reads.
bool tvs_usable(int V, int es, int gamma) {
    if (tuning().tv_kernel == MTP_KERNEL_RESIDENT) return false;  // a TMEM request that does not fit streams
    return gamma <= tvs_max_gamma() && V % (16 / es) == 0;
}

bool plan_tvs(int dev, int dtype, int V, int es, int gamma, int units, Plan &p, bool topk = false) {
    const mtp_tuning tu = tuning();
    const int forced = tuned_cluster(tu);
    int R = tu.ring_slots;
    if (R < 2 || R > stream_max_ring()) R = 2;
    const int l2mb = tu.tv_l2_mb;
    const double pos_bytes = 2.0 * gamma * static_cast<double>(V) * es;
    int cap_l2 = l2mb > 0 ? static_cast<int>((static_cast<double>(l2mb) * 1048576.0) / pos_bytes) : 1 << 30;
    if (cap_l2 < 1) cap_l2 = 1;
    const uint32_t cap = smem_optin(dev);
    const int nw = tvs_threads() / 32;
    const int nv = V / (16 / es);
    long best = -1;
    bool found = false;
    for (int C = 1; C <= MAX_C; C *= 2) {
        if (forced && C != forced) continue;
        const int S = C * nw;
        if (S > tvs_max_segments()) continue;
        const int nvs = (nv + S - 1) / S;
        const int cv = stream_chunk_for(nvs, 3);
        const uint32_t smem = tvs_hdr_bytes() + tvs_rec_bytes(gamma, S) + tvs_bits_bytes(gamma, nvs) +
                              static_cast<uint32_t>(nw * R) * stream_slot_bytes(cv);
        if (smem > cap) continue;
        const void *func = tvs_kernel(dtype, cv, topk);
        if (prepare_func(dev, func) != cudaSuccess) return false;
        const int nc = max_clusters(dev, func, C, smem, tvs_threads());
        if (nc <= 0) continue;
        int used = nc < units ? nc : units;
        if (used > cap_l2) used = cap_l2;
        if (tu.max_clusters > 0 && used > tu.max_clusters) used = tu.max_clusters;
        const long warps = static_cast<long>(used) * C * nw;
        // the most warps in flight; within 5 % the larger cluster
        if (!found || warps * 20 > best * 21 || (warps * 21 >= best * 20 && C > p.C)) {
            if (warps > best) best = warps;
            p = Plan{};
            p.C = C;
            p.smem = smem;
            p.clusters = used;
            p.threads = tvs_threads();
            p.ring = R;
            p.seg_vectors = nvs;
            p.cv = cv;
            p.func = func;
            found = true;
        }
    }
    return found;
}

// TMEM-resident TV kernel: clusters of C CTAs x 16 warps, one CTA per SM
// holding all 512 TMEM columns, in which its warps park their segments of
// the position's gamma draft rows (NS 16-byte vectors per lane and row, 4
// columns each, 128 columns per warp).  The warps of a CTA form teams that
// work on different positions; a segment is 1 / (C x team warps) of a row.  The smallest power-of-two C whose
// segments fit wins (the most positions in flight).  TMEM allocation blocks
// until columns are free, so the shared memory asked for keeps a second CTA
// off the SM: more than half of the SM's shared memory.
bool tvm_usable(int V, int es, int gamma) {
    const int k = tuning().tv_kernel;
    if (k == MTP_KERNEL_STREAM || k == MTP_KERNEL_RESIDENT) return false;
    return gamma <= tvm_max_gamma() && V % (16 / es) == 0;
}

bool plan_tvm(int dev, int dtype, int V, int es, int gamma, int units, Plan &p) {
    const mtp_tuning tu = tuning();
    const int forced = tuned_cluster(tu);
    int per_sm = 0, reserved = 0;
    if (cudaDeviceGetAttribute(&per_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&reserved, cudaDevAttrReservedSharedMemoryPerBlock, dev) != cudaSuccess) {
        (void)cudaGetLastError();
        return false;
    }
    const uint32_t hi = smem_optin(dev);
    const uint32_t lo = static_cast<uint32_t>(per_sm / 2 - reserved + 128) & ~127u;  // 2 CTAs do not fit
    const int nv = V / (16 / es);
    const int ns_set[] = {2, 4, 5, 8, 10};
    for (int C = 1; C <= tvm_max_cluster(); C *= 2) {
        if (forced && C != forced) continue;
        const int S = C * tvm_team_warps();
        const int nvs = (nv + S - 1) / S;
        const int need = (nvs + 31) / 32;
        int ns = 0;
        for (int c : ns_set)
            if (c >= need) {
                ns = c;
                break;
            }
        if (!ns || gamma * ns * 4 > tvm_warp_cols()) continue;
        int R = tu.ring_slots;
        if (R < 2 || R > tvm_max_ring()) R = tvm_max_ring();
        while (R >= 2 && tvm_smem_bytes(gamma, C, ns, R) > hi) --R;
        if (R < 2) continue;
        uint32_t smem = tvm_smem_bytes(gamma, C, ns, R);
        if (smem < lo) smem = lo;  // padding: keeps a second CTA (and its TMEM allocation) off the SM
        if (smem > hi || lo > hi) continue;
        const void *func = tvm_kernel(dtype, ns);
        if (!func) continue;
        if (prepare_func(dev, func) != cudaSuccess) return false;
        const int nc = max_clusters(dev, func, C, smem, tvm_threads());
        if (nc <= 0) continue;
        // every cluster takes tvm_teams() positions at a time
        const int want = (units + tvm_teams() - 1) / tvm_teams();
        int used = nc < want ? nc : want;
        if (tu.max_clusters > 0 && used > tu.max_clusters) used = tu.max_clusters;
        p = Plan{};
        p.C = C;
        p.smem = smem;
        p.clusters = used;
        p.threads = tvm_threads();
        p.ring = R;
        p.seg_vectors = nvs;
        p.nres = gamma;  // every draft row of a position stays on chip
        p.func = func;
        return true;
    }
    return false;
}

// TMEM-resident row-statistics kernel: clusters of C CTAs x 16 warps, one
// CTA per SM holding all 512 TMEM columns; a warp parks two draft row
// segments at a time (NS vectors per lane each).  The smallest C whose
// segments fit wins; shared memory above half the SM's keeps a second CTA
// (and its TMEM allocation) off the SM.
bool stm_usable(int V, int es, int gamma) {
    // measured slower than the cluster-resident kernel on the B = 256, gamma
    // = 7 fp32 rows (each warp's chain of exchanges per sequence is latency
    // bound with one CTA per SM): on request only
    if (tuning().stats_kernel != MTP_KERNEL_TMEM) return false;
    return gamma <= stm_max_gamma() && V % (16 / es) == 0;
}

bool plan_stm(int dev, int dtype, int V, int es, int gamma, int units, Plan &p) {
    const mtp_tuning tu = tuning();
    const int forced = tuned_cluster(tu);
    int per_sm = 0, reserved = 0;
    if (cudaDeviceGetAttribute(&per_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&reserved, cudaDevAttrReservedSharedMemoryPerBlock, dev) != cudaSuccess) {
        (void)cudaGetLastError();
        return false;
    }
    const uint32_t hi = smem_optin(dev);
    const uint32_t lo = static_cast<uint32_t>(per_sm / 2 - reserved + 128) & ~127u;  // 2 CTAs do not fit
    const int nv = V / (16 / es);
    const int ns_set[] = {2, 4, 5, 8, 10, 15};
    for (int C = 1; C <= stm_max_cluster(); C *= 2) {
        if (forced && C != forced) continue;
        const int S = C * (stm_threads() / 32);
        const int nvs = (nv + S - 1) / S;
        const int need = (nvs + 31) / 32;
        int ns = 0;
        for (int c : ns_set)
            if (c >= need) {
                ns = c;
                break;
            }
        if (!ns || stm_parked() * ns * 4 > stm_warp_cols()) continue;
        int R = tu.ring_slots;
        if (R < 2 || R > stm_max_ring()) R = stm_max_ring();
        while (R >= 2 && stm_smem_bytes(gamma, C, ns, R) > hi) --R;
        if (R < 2) continue;
        uint32_t smem = stm_smem_bytes(gamma, C, ns, R);
        if (smem < lo) smem = lo;  // padding: keeps a second CTA (and its TMEM allocation) off the SM
        if (smem > hi) continue;
        const void *func = stm_kernel(dtype, ns);
        if (!func) continue;
        if (prepare_func(dev, func) != cudaSuccess) return false;
        const int nc = max_clusters(dev, func, C, smem, stm_threads());
        if (nc <= 0) continue;
        int used = nc < units ? nc : units;
        if (tu.max_clusters > 0 && used > tu.max_clusters) used = tu.max_clusters;
        p = Plan{};
        p.C = C;
        p.smem = smem;
        p.clusters = used;
        p.threads = stm_threads();
        p.ring = R;
        p.seg_vectors = nvs;
        p.nres = stm_parked();
        p.func = func;
        return true;
    }
    return false;
}

// Persistent TV kernel: two target slots, nres (>= 2, ideally gamma) draft
// slots and gamma rows of indicator bits per CTA.
bool plan_tv(int dev, const void *func, int V, int es, int gamma, int units, Plan &p) {
    const mtp_tuning tu = tuning();
    const int forced = tu.cluster_size;
    const int cap_nres = tu.tv_resident_drafts;
    const uint32_t cap = smem_optin(dev);
    long best = -1;
    for (int C = 1; C <= MAX_C; ++C) {
        if (forced && C != forced) continue;
        const uint32_t sb = slice_buffer_bytes(V, es, C);
        const uint32_t bitb = static_cast<uint32_t>(gamma) * static_cast<uint32_t>(slice_vectors(V, 16 / es, C));
        const uint32_t fixed = tv_hdr_bytes() + 2 * sb + ((bitb + 127u) & ~127u);
        if (fixed + sb > cap) continue;
        int nres = static_cast<int>((cap - fixed) / sb);
        if (nres > gamma) nres = gamma;
        if (cap_nres > 0 && nres > cap_nres) nres = cap_nres;
        if (nres < 1) continue;
        // with every draft resident, prefer the smallest footprint that holds them
        const uint32_t smem = fixed + static_cast<uint32_t>(nres) * sb;
        const int nc = max_clusters(dev, func, C, smem, tv_threads());
        if (nc <= 0) continue;
        const int used = nc < units ? nc : units;
        // working CTAs, with a penalty for draft slices re-read in the epilogue
        const long score = static_cast<long>(used) * C * (nres == gamma ? 2 : 1);
        if (score > best) {
            best = score;
            p = {C, sb, smem, nres, used, 1, tv_threads()};
        }
    }
    return best > 0;
}

int launch(const void *func, const Plan &p, void *args, mtp_stream_t stream) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(p.clusters) * static_cast<unsigned>(p.C));
    cfg.blockDim = dim3(p.threads);
    cfg.dynamicSmemBytes = p.smem;
    cfg.stream = reinterpret_cast<cudaStream_t>(stream);
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = p.C;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    // programmatic stream serialization: the kernel may start while the
    // previous launch on the stream finishes; it waits for it in-kernel
    // (griddepcontrol.wait) before touching global memory
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = p.pdl ? 2 : 1;
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
    const int es = esize(dtype);
    const void *func = nullptr;
    Plan p;
    if (mode == MODE_VERIFY && stream_usable(V, es, gamma)) {
        if (plan_stream(dev, dtype == MTP_DTYPE_F32 ? 0 : 1, V, es, gamma, B, p)) func = p.func;
    }
    if (!func) {
        func = row_kernel(dtype == MTP_DTYPE_F32 ? 0 : 1, mode);
        if (prepare_func(dev, func) != cudaSuccess) return MTP_ERR_CUDA;
        if (!plan_row(dev, func, V, es, B, p)) return MTP_ERR_NO_DEVICE;
    }
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
    A.streams = p.streams;
    A.ring = p.ring;
    A.depth = p.depth;
    A.seg_vectors = p.seg_vectors;
    A.tokens = tokens;
    A.accept_len = accept_len;
    A.alpha = alpha;
    A.entropy = entropy;
    A.flags = flags;
    A.yhat = nullptr;
    return launch(func, p, &A, stream);
}

// Streaming row-pair statistics kernel (diagnostics; row statistics on
// request): clusters of C CTAs x NT/32 warps, one vocabulary segment per
// warp, one sequence per cluster at a time.  Same rule as the streaming TV
// kernel: the most warps in flight, within 5 % the larger cluster;
// mtp_tuning.pair_l2_mb caps the sequences in flight by the bytes of the row
// pairs they re-read.  Measured on GB300 at B = 256, gamma = 7, V = 151,936
// fp32, the cluster-resident kernel (one load per row, the second pass from
// shared memory) computes the row statistics faster than this kernel, whose
// second pass re-reads rows that L2 no longer holds; mtp_row_stats therefore
// uses it only when mtp_tuning.stats_kernel asks for it.
bool pairs_usable(int V, int es, int gamma) {
    return gamma <= pair_max_gamma() && V % (16 / es) == 0;
}

bool stats_streamed() { return tuning().stats_kernel == MTP_KERNEL_STREAM; }

bool plan_pairs(int dev, int dtype, int V, int es, int gamma, int units, int mode, Plan &p) {
    const mtp_tuning tu = tuning();
    const int forced = tuned_cluster(tu);
    int R = tu.ring_slots;
    if (R < 2 || R > pair_max_ring()) R = 2;
    const int l2mb = tu.pair_l2_mb;
    const double seq_bytes = 2.0 * static_cast<double>(V) * es;  // the row pair a sequence re-reads next
    int cap_l2 = l2mb > 0 ? static_cast<int>((static_cast<double>(l2mb) * 1048576.0) / seq_bytes) : 1 << 30;
    if (cap_l2 < 1) cap_l2 = 1;
    const uint32_t cap = smem_optin(dev);
    const int nw = pair_threads() / 32;
    const int nv = V / (16 / es);
    long best = -1;
    bool found = false;
    for (int C = 1; C <= MAX_C; C *= 2) {
        if (forced && C != forced) continue;
        const int S = C * nw;
        if (S > pair_max_segments()) continue;
        const int nvs = (nv + S - 1) / S;
        int cv = stream_chunk_for(nvs, 4);
        if (mode == PAIR_DIAG && cv == 192) cv = 128;  // the 3 KB diagnostics variant spills
        const uint32_t smem = pair_hdr_bytes() + pair_rec_bytes(gamma, S, mode) +
                              static_cast<uint32_t>(nw * R) * stream_slot_bytes(cv);
        if (smem > cap) continue;
        const void *func = pair_kernel(dtype, cv, mode);
        if (prepare_func(dev, func) != cudaSuccess) return false;
        const int nc = max_clusters(dev, func, C, smem, pair_threads());
        if (nc <= 0) continue;
        int used = nc < units ? nc : units;
        if (used > cap_l2) used = cap_l2;
        if (tu.max_clusters > 0 && used > tu.max_clusters) used = tu.max_clusters;
        const long warps = static_cast<long>(used) * C * nw;
        if (!found || warps * 20 > best * 21 || (warps * 21 >= best * 20 && C > p.C)) {
            if (warps > best) best = warps;
            p = Plan{};
            p.C = C;
            p.smem = smem;
            p.clusters = used;
            p.threads = pair_threads();
            p.ring = R;
            p.seg_vectors = nvs;
            p.cv = cv;
            p.func = func;
            found = true;
        }
    }
    return found;
}

int pair_call(int mode, const void *target, const void *draft, mtp_dtype dtype, const float *temp, int B,
              int gamma, int V, float *alpha, float *ent_p, float *ent_q, float *kl, int32_t *yhat, float *p_yhat,
              int32_t *rs_better, int32_t *flags, mtp_stream_t stream) {
    int dev;
    if (current_device(dev) != MTP_OK) return MTP_ERR_CUDA;
    const int es = esize(dtype);
    Plan p;
    if (!plan_pairs(dev, dtype == MTP_DTYPE_F32 ? 0 : 1, V, es, gamma, B, mode, p)) return MTP_ERR_NO_DEVICE;
    PairArgs A = {};
    A.target = target;
    A.draft = draft;
    A.temp = temp;
    A.B = B;
    A.gamma = gamma;
    A.V = V;
    A.ring = p.ring;
    A.seg_vectors = p.seg_vectors;
    A.alpha = alpha;
    A.ent_p = ent_p;
    A.ent_q = ent_q;
    A.kl = kl;
    A.yhat = yhat;
    A.p_yhat = p_yhat;
    A.rs_better = rs_better;
    A.flags = flags;
    return launch(p.func, p, &A, stream);
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

extern "C" int mtp_to_verify(const void *target_logits, const void *draft_logits, mtp_dtype dtype,
                             const float *temperature, const float *uniforms, int B, int gamma, int V,
                             int32_t *out_tokens, int32_t *accept_len, int32_t *draft_tokens, int32_t *row_flags,
                             mtp_stream_t stream) {
    if (dtype != MTP_DTYPE_F32 && dtype != MTP_DTYPE_BF16) return MTP_ERR_UNSUPPORTED_DTYPE;
    if (B < 0 || gamma < 1 || gamma > MTP_MAX_GAMMA || V < 1) return MTP_ERR_INVALID_ARG;
    if (B == 0) return MTP_OK;
    if (!target_logits || !draft_logits || !temperature || !uniforms || !out_tokens || !accept_len)
        return MTP_ERR_INVALID_ARG;
    if (!aligned16(target_logits) || !aligned16(draft_logits)) return MTP_ERR_MISALIGNED;
    const int es = esize(dtype);
    // the streaming kernel serves target-only verification: whole 16-byte
    // vectors per row and gamma up to its limit
    if (V % (16 / es) != 0) return MTP_ERR_MISALIGNED;
    if (gamma > stream_max_gamma()) return MTP_ERR_INVALID_ARG;
    int dev;
    if (current_device(dev) != MTP_OK) return MTP_ERR_CUDA;
    Plan p;
    if (!plan_stream(dev, dtype == MTP_DTYPE_F32 ? 0 : 1, V, es, gamma, B, p, 1)) return MTP_ERR_NO_DEVICE;
    VerifyArgs A = {};
    A.target = target_logits;
    A.draft = draft_logits;
    A.ids = nullptr;
    A.temp = temperature;
    A.unif = uniforms;
    A.B = B;
    A.gamma = gamma;
    A.V = V;
    A.aligned = 1;
    A.streams = 1;
    A.ring = p.ring;
    A.depth = p.depth;
    A.seg_vectors = p.seg_vectors;
    A.tokens = out_tokens;
    A.accept_len = accept_len;
    A.flags = row_flags;
    A.yhat = draft_tokens;
    return launch(p.func, p, &A, stream);
}

extern "C" int mtp_gumbel_verify(const void *target_logits, const void *draft_logits, mtp_dtype dtype,
                                 const int32_t *draft_ids, const float *temperature, const float *uniforms,
                                 uint64_t seed, uint32_t offset, int B, int gamma, int V, int32_t *out_tokens,
                                 int32_t *accept_len, int32_t *row_flags, mtp_stream_t stream) {
    if (dtype != MTP_DTYPE_F32 && dtype != MTP_DTYPE_BF16) return MTP_ERR_UNSUPPORTED_DTYPE;
    if (B < 0 || gamma < 1 || gamma > MTP_MAX_GAMMA || V < 1) return MTP_ERR_INVALID_ARG;
    if (B == 0) return MTP_OK;
    if (!target_logits || !draft_logits || !draft_ids || !temperature || !uniforms || !out_tokens || !accept_len)
        return MTP_ERR_INVALID_ARG;
    if (!aligned16(target_logits) || !aligned16(draft_logits)) return MTP_ERR_MISALIGNED;
    const int es = esize(dtype);
    // the streaming kernel serves the Gumbel-max variant: whole 16-byte
    // vectors per row and gamma up to its limit
    if (V % (16 / es) != 0) return MTP_ERR_MISALIGNED;
    if (gamma > stream_max_gamma()) return MTP_ERR_INVALID_ARG;
    int dev;
    if (current_device(dev) != MTP_OK) return MTP_ERR_CUDA;
    Plan p;
    if (!plan_stream(dev, dtype == MTP_DTYPE_F32 ? 0 : 1, V, es, gamma, B, p, 2)) return MTP_ERR_NO_DEVICE;
    VerifyArgs A = {};
    A.target = target_logits;
    A.draft = draft_logits;
    A.ids = draft_ids;
    A.temp = temperature;
    A.unif = uniforms;
    A.B = B;
    A.gamma = gamma;
    A.V = V;
    A.aligned = 1;
    A.streams = 1;
    A.ring = p.ring;
    A.depth = p.depth;
    A.seg_vectors = p.seg_vectors;
    A.tokens = out_tokens;
    A.accept_len = accept_len;
    A.flags = row_flags;
    A.yhat = nullptr;
    A.seed_lo = static_cast<uint32_t>(seed);
    A.seed_hi = static_cast<uint32_t>(seed >> 32);
    A.offset = offset;
    return launch(p.func, p, &A, stream);
}

extern "C" int mtp_draft_sample(const void *draft_logits, mtp_dtype dtype, const float *temperature,
                                const float *uniforms, int method, uint64_t seed, uint32_t offset, int R, int V,
                                int32_t *out_ids, int32_t *row_flags, mtp_stream_t stream) {
    if (dtype != MTP_DTYPE_F32 && dtype != MTP_DTYPE_BF16) return MTP_ERR_UNSUPPORTED_DTYPE;
    if (R < 0 || V < 1 || (method != 0 && method != 1)) return MTP_ERR_INVALID_ARG;
    if (R == 0) return MTP_OK;
    if (!draft_logits || !temperature || !out_ids || (method == 0 && !uniforms)) return MTP_ERR_INVALID_ARG;
    if (!aligned16(draft_logits)) return MTP_ERR_MISALIGNED;
    const int es = esize(dtype);
    if (V % (16 / es) != 0) return MTP_ERR_MISALIGNED;
    int dev;
    if (current_device(dev) != MTP_OK) return MTP_ERR_CUDA;
    Plan p;
    // Gumbel-max: one pass per row (no normaliser needed), clusters of at
    // most 8; a forced larger cluster takes the streaming kernel below
    if (method == 1 && plan_gsample(dev, dtype == MTP_DTYPE_F32 ? 0 : 1, V, es, R, p)) {
        VerifyArgs A = {};
        A.target = draft_logits;
        A.temp = temperature;
        A.B = R;
        A.V = V;
        A.aligned = 1;
        A.tokens = out_ids;
        A.flags = row_flags;
        A.seed_lo = static_cast<uint32_t>(seed);
        A.seed_hi = static_cast<uint32_t>(seed >> 32);
        A.offset = offset;
        return launch(p.func, p, &A, stream);
    }
    // each row is a one-row sequence of the streaming verify kernel: no draft
    // step, and its final draw (the bonus) samples the row
    const int mode = method == 0 ? 0 : 2;
    if (!plan_stream(dev, dtype == MTP_DTYPE_F32 ? 0 : 1, V, es, 0, R, p, mode, true)) return MTP_ERR_NO_DEVICE;
    VerifyArgs A = {};
    A.target = draft_logits;
    A.draft = draft_logits;
    A.ids = nullptr;
    A.temp = temperature;
    A.unif = method == 0 ? uniforms : nullptr;
    A.B = R;
    A.gamma = 0;
    A.V = V;
    A.aligned = 1;
    A.streams = 1;
    A.ring = p.ring;
    A.depth = 0;
    A.seg_vectors = p.seg_vectors;
    A.tokens = out_ids;
    A.accept_len = nullptr;
    A.flags = row_flags;
    A.yhat = nullptr;
    A.seed_lo = static_cast<uint32_t>(seed);
    A.seed_hi = static_cast<uint32_t>(seed >> 32);
    A.offset = offset;
    return launch(p.func, p, &A, stream);
}

extern "C" int mtp_row_stats(const void *target_logits, const void *draft_logits, mtp_dtype dtype,
                             const float *temperature, int B, int gamma, int V, float *alpha, float *entropy,
                             int32_t *row_flags, mtp_stream_t stream) {
    if (B > 0 && (!alpha || !entropy)) return MTP_ERR_INVALID_ARG;
    if (dtype != MTP_DTYPE_F32 && dtype != MTP_DTYPE_BF16) return MTP_ERR_UNSUPPORTED_DTYPE;
    if (B > 0 && gamma >= 1 && gamma <= MTP_MAX_GAMMA && V >= 1 && target_logits && draft_logits && temperature &&
        aligned16(target_logits) && aligned16(draft_logits) && stm_usable(V, esize(dtype), gamma)) {
        int dev;
        if (current_device(dev) != MTP_OK) return MTP_ERR_CUDA;
        Plan p;
        if (plan_stm(dev, dtype == MTP_DTYPE_F32 ? 0 : 1, V, esize(dtype), gamma, B, p)) {
            VerifyArgs A = {};
            A.target = target_logits;
            A.draft = draft_logits;
            A.temp = temperature;
            A.B = B;
            A.gamma = gamma;
            A.V = V;
            A.aligned = 1;
            A.ring = p.ring;
            A.seg_vectors = p.seg_vectors;
            A.alpha = alpha;
            A.entropy = entropy;
            A.flags = row_flags;
            return launch(p.func, p, &A, stream);
        }
    }
    if (B > 0 && gamma >= 1 && V >= 1 && target_logits && draft_logits && temperature && aligned16(target_logits) &&
        aligned16(draft_logits) && stats_streamed() && pairs_usable(V, esize(dtype), gamma))
        return pair_call(PAIR_STATS, target_logits, draft_logits, dtype, temperature, B, gamma, V, alpha, entropy,
                         nullptr, nullptr, nullptr, nullptr, nullptr, row_flags, stream);
    return row_call(MODE_STATS, target_logits, draft_logits, dtype, nullptr, temperature, nullptr, B, gamma, V,
                    nullptr, nullptr, alpha, entropy, row_flags, stream);
}

extern "C" int mtp_rs_diagnostics(const void *target_logits, const void *draft_logits, mtp_dtype dtype,
                                  const float *temperature, int B, int gamma, int V, float *alpha, float *ent_p,
                                  float *ent_q, float *kl, int32_t *yhat, float *p_yhat, int32_t *rs_better,
                                  int32_t *row_flags, mtp_stream_t stream) {
    if (dtype != MTP_DTYPE_F32 && dtype != MTP_DTYPE_BF16) return MTP_ERR_UNSUPPORTED_DTYPE;
    if (B < 0 || gamma < 1 || gamma > pair_max_gamma() || V < 1) return MTP_ERR_INVALID_ARG;
    if (B == 0) return MTP_OK;
    if (!target_logits || !draft_logits || !temperature) return MTP_ERR_INVALID_ARG;
    const int es = esize(dtype);
    if (!aligned16(target_logits) || !aligned16(draft_logits) || V % (16 / es) != 0) return MTP_ERR_MISALIGNED;
    return pair_call(PAIR_DIAG, target_logits, draft_logits, dtype, temperature, B, gamma, V, alpha, ent_p, ent_q,
                     kl, yhat, p_yhat, rs_better, row_flags, stream);
}

extern "C" int mtp_tv_loss_ex(const void *target_logits, const void *draft_logits, mtp_dtype dtype,
                              float temperature, int N, int gamma, int V, float grad_scale, int target_layout,
                              int loss_kind, float tau_max, float *loss, float *alpha, float *grad_draft_logits,
                              int32_t *row_flags, mtp_stream_t stream) {
    if (dtype != MTP_DTYPE_F32 && dtype != MTP_DTYPE_BF16) return MTP_ERR_UNSUPPORTED_DTYPE;
    if (N < 0 || gamma < 1 || gamma > MTP_MAX_GAMMA || V < 1) return MTP_ERR_INVALID_ARG;
    if ((target_layout != 0 && target_layout != 1) || (loss_kind != 0 && loss_kind != 1)) return MTP_ERR_INVALID_ARG;
    if (loss_kind == 1 && !(tau_max >= 0.f)) return MTP_ERR_INVALID_ARG;
    if (N == 0) return MTP_OK;
    if (!target_logits || !draft_logits || !loss || !grad_draft_logits) return MTP_ERR_INVALID_ARG;
    if (!aligned16(target_logits) || !aligned16(draft_logits) || !aligned16(grad_draft_logits))
        return MTP_ERR_MISALIGNED;
    int dev;
    if (current_device(dev) != MTP_OK) return MTP_ERR_CUDA;
    const int es = esize(dtype);
    const int d = dtype == MTP_DTYPE_F32 ? 0 : 1;
    const void *func = nullptr;
    Plan p;
    if (tvm_usable(V, es, gamma) && plan_tvm(dev, d, V, es, gamma, N, p)) func = p.func;
    if (!func && tvs_usable(V, es, gamma) && plan_tvs(dev, d, V, es, gamma, N, p)) func = p.func;
    if (!func) {
        func = tv_kernel(d);
        if (prepare_func(dev, func) != cudaSuccess) return MTP_ERR_CUDA;
        if (!plan_tv(dev, func, V, es, gamma, N, p)) return MTP_ERR_NO_DEVICE;
    }
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
    A.ring = p.ring;
    A.seg_vectors = p.seg_vectors;
    A.loss = loss;
    A.alpha = alpha;
    A.grad = grad_draft_logits;
    A.flags = row_flags;
    A.shared_target = target_layout;
    A.loss_kind = loss_kind;
    A.tau_max = loss_kind == 1 ? tau_max : 0.f;
    A.topk_idx = nullptr;
    A.K = 0;
    A.grad32 = (reinterpret_cast<uintptr_t>(grad_draft_logits) & 31u) == 0 ? 1 : 0;
    const mtp_tuning tu = tuning();
    A.wait_ns = tu.fault_wait_us > 0 ? static_cast<uint32_t>(tu.fault_wait_us) * 1000u : 0u;
    A.skip_t = tu.fault_skip_position > 0 ? tu.fault_skip_position - 1 : -1;
    return launch(func, p, &A, stream);
}

extern "C" int mtp_tv_loss_topk(const void *target_values, const int32_t *target_idx, const void *draft_logits,
                                mtp_dtype dtype, float temperature, int N, int gamma, int K, int V, float grad_scale,
                                int loss_kind, float tau_max, float *loss, float *alpha, float *grad_draft_logits,
                                int32_t *row_flags, mtp_stream_t stream) {
    if (dtype != MTP_DTYPE_F32 && dtype != MTP_DTYPE_BF16) return MTP_ERR_UNSUPPORTED_DTYPE;
    if (N < 0 || gamma < 1 || gamma > MTP_MAX_GAMMA || V < 1 || K < 1 || K > V) return MTP_ERR_INVALID_ARG;
    if (loss_kind != 0 && loss_kind != 1) return MTP_ERR_INVALID_ARG;
    if (loss_kind == 1 && !(tau_max >= 0.f)) return MTP_ERR_INVALID_ARG;
    if (N == 0) return MTP_OK;
    if (!target_values || !target_idx || !draft_logits || !loss || !grad_draft_logits) return MTP_ERR_INVALID_ARG;
    const int es = esize(dtype);
    if (!aligned16(draft_logits) || !aligned16(grad_draft_logits) || V % (16 / es) != 0) return MTP_ERR_MISALIGNED;
    // the streaming TV kernel serves the top-K target: gamma up to its limit
    if (gamma > tvs_max_gamma()) return MTP_ERR_INVALID_ARG;
    int dev;
    if (current_device(dev) != MTP_OK) return MTP_ERR_CUDA;
    Plan p;
    if (!plan_tvs(dev, dtype == MTP_DTYPE_F32 ? 0 : 1, V, es, gamma, N, p, true)) return MTP_ERR_NO_DEVICE;
    TVArgs A = {};
    A.target = target_values;
    A.draft = draft_logits;
    A.temperature = temperature;
    A.grad_scale = grad_scale;
    A.N = N;
    A.gamma = gamma;
    A.V = V;
    A.aligned = 1;
    A.ring = p.ring;
    A.seg_vectors = p.seg_vectors;
    A.loss = loss;
    A.alpha = alpha;
    A.grad = grad_draft_logits;
    A.flags = row_flags;
    A.shared_target = 0;
    A.loss_kind = loss_kind;
    A.tau_max = loss_kind == 1 ? tau_max : 0.f;
    A.topk_idx = target_idx;
    A.K = K;
    A.grad32 = (reinterpret_cast<uintptr_t>(grad_draft_logits) & 31u) == 0 ? 1 : 0;
    A.wait_ns = 0;
    A.skip_t = -1;
    return launch(p.func, p, &A, stream);
}

extern "C" int mtp_tv_loss_fwd_bwd(const void *target_logits, const void *draft_logits, mtp_dtype dtype,
                                   float temperature, int N, int gamma, int V, float grad_scale, float *loss,
                                   float *alpha, float *grad_draft_logits, int32_t *row_flags,
                                   mtp_stream_t stream) {
    return mtp_tv_loss_ex(target_logits, draft_logits, dtype, temperature, N, gamma, V, grad_scale, 0, 0, 0.f, loss,
                          alpha, grad_draft_logits, row_flags, stream);
}

extern "C" int mtp_query_plan(int op, mtp_dtype dtype, int units, int gamma, int V, int *cluster_size,
                              int *clusters, int *smem_bytes, int *resident_drafts) {
    if (dtype != MTP_DTYPE_F32 && dtype != MTP_DTYPE_BF16) return MTP_ERR_UNSUPPORTED_DTYPE;
    if (op < 0 || op > 11 || units < 1 || gamma < 1 || gamma > MTP_MAX_GAMMA || V < 1) return MTP_ERR_INVALID_ARG;
    int dev;
    if (current_device(dev) != MTP_OK) return MTP_ERR_CUDA;
    const int d = dtype == MTP_DTYPE_F32 ? 0 : 1;
    const int es = esize(dtype);
    Plan p;
    bool ok = false, streamed = false;
    if (op == 0 && stream_usable(V, es, gamma)) ok = streamed = plan_stream(dev, d, V, es, gamma, units, p);
    if (op == 3 && tvm_usable(V, es, gamma)) ok = plan_tvm(dev, d, V, es, gamma, units, p);
    if (op == 3 && !ok && tvs_usable(V, es, gamma)) ok = streamed = plan_tvs(dev, d, V, es, gamma, units, p);
    if (op == 2 && stm_usable(V, es, gamma)) ok = plan_stm(dev, d, V, es, gamma, units, p);
    if (op == 2 && !ok && stats_streamed() && pairs_usable(V, es, gamma)) ok = streamed = plan_pairs(dev, d, V, es, gamma, units, PAIR_STATS, p);
    if (op == 10) {  // draft sampling by inverse CDF: one-row sequences of the streaming kernel
        if (V % (16 / es) != 0) return MTP_ERR_INVALID_ARG;
        ok = streamed = plan_stream(dev, d, V, es, 0, units, p, 0, true);
        if (!ok) return MTP_ERR_NO_DEVICE;
    }
    if (op == 11) {  // draft sampling by Gumbel-max: the one-pass kernel, else the streaming kernel
        if (V % (16 / es) != 0) return MTP_ERR_INVALID_ARG;
        ok = plan_gsample(dev, d, V, es, units, p);
        if (!ok) ok = streamed = plan_stream(dev, d, V, es, 0, units, p, 2, true);
        if (!ok) return MTP_ERR_NO_DEVICE;
    }
    if (op == 8 || op == 9) {  // target-only verify, Gumbel-max verify: streaming kernel only
        if (gamma > stream_max_gamma() || V % (16 / es) != 0) return MTP_ERR_INVALID_ARG;
        ok = streamed = plan_stream(dev, d, V, es, gamma, units, p, op == 8 ? 1 : 2);
        if (!ok) return MTP_ERR_NO_DEVICE;
    }
    if (op == 6) {
        if (gamma > pair_max_gamma() || V % (16 / es) != 0) return MTP_ERR_INVALID_ARG;
        ok = streamed = plan_pairs(dev, d, V, es, gamma, units, PAIR_DIAG, p);
        if (!ok) return MTP_ERR_NO_DEVICE;
    }
    if (!ok) {
        const int mode = (op == 0 || op == 4) ? MODE_VERIFY : op == 1 ? MODE_VERIFY_STATS : MODE_STATS;
        const bool tv = op == 3 || op == 5;
        const void *func = tv ? tv_kernel(d) : row_kernel(d, mode);
        if (prepare_func(dev, func) != cudaSuccess) return MTP_ERR_CUDA;
        ok = tv ? plan_tv(dev, func, V, es, gamma, units, p) : plan_row(dev, func, V, es, units, p);
    }
    if (!ok) return MTP_ERR_NO_DEVICE;
    if (streamed) p.nres = (op == 0 || op >= 8) ? p.ring : 0;
    if (cluster_size) *cluster_size = p.C;
    if (clusters) *clusters = p.clusters;
    if (smem_bytes) *smem_bytes = static_cast<int>(p.smem);
    if (resident_drafts) *resident_drafts = p.nres;
    return MTP_OK;
}

extern "C" int mtp_set_tuning(const mtp_tuning *t) {
    std::lock_guard<std::mutex> lk(g_mu);
    if (t) g_tune = *t;
    else g_tune = mtp_tuning{};
    return MTP_OK;
}

extern "C" int mtp_get_tuning(mtp_tuning *t) {
    if (!t) return MTP_ERR_INVALID_ARG;
    std::lock_guard<std::mutex> lk(g_mu);
    *t = g_tune;
    return MTP_OK;
}

extern "C" const char *mtp_status_string(int status) {
    switch (status) {
        case MTP_OK: return "ok";
        case MTP_ERR_INVALID_ARG: return "invalid argument";
        case MTP_ERR_UNSUPPORTED_DTYPE: return "unsupported dtype";
        case MTP_ERR_MISALIGNED: return "logit or gradient base pointer not 16-byte aligned";
        case MTP_ERR_CUDA: return "CUDA error";
        case MTP_ERR_TIMEOUT: return "an on-chip wait gave up (rows flagged MTP_ROW_TIMEOUT)";
        case MTP_ERR_NO_DEVICE: return "no usable cluster launch configuration on this device";
        default: return "unknown status";
    }
}
