// kernels.h -- internal interface between the C-ABI layer and the kernels.
#pragma once

#include <stdint.h>

namespace mtp {

constexpr int MAX_GAMMA = 32;

// Kernel modes of the row kernel.
enum RowMode { MODE_VERIFY = 0, MODE_VERIFY_STATS = 1, MODE_STATS = 2 };

struct VerifyArgs {
    const void *target;  // [B, gamma+1, V]
    const void *draft;   // [B, gamma, V]
    const int32_t *ids;  // [B, gamma]          (verify modes)
    const float *temp;   // [B]
    const float *unif;   // [B, gamma+1]        (verify modes)
    int B, gamma, V;
    int aligned;            // every row starts on 16 bytes and V is whole vectors
    uint32_t slice_bytes;   // shared bytes of one row slice
    int streams;            // sequences in flight per CTA (1 or 2)
    int ring;               // streaming kernel: chunk slots per warp
    int depth;              // streaming kernel: positions streamed ahead of the last decision
    int seg_vectors;        // streaming kernel: 16-byte vectors per warp segment
    int32_t *tokens;        // [B, gamma+1]      (verify modes)
    int32_t *accept_len;    // [B]               (verify modes)
    float *alpha;           // [B, gamma]        (stats modes)
    float *entropy;         // [B, gamma+1]      (stats modes)
    int32_t *flags;         // [B] or null
    int32_t *yhat;          // [B, gamma] or null (target-only: the arg max draft tokens)
    uint32_t seed_lo, seed_hi, offset;  // Gumbel-max final draw: noise stream key and counter word
};

struct TVArgs {
    const void *target;  // [N, gamma, V]
    const void *draft;   // [N, gamma, V]
    float temperature, grad_scale;
    int N, gamma, V;
    int aligned;
    int nres;               // draft slices kept on chip (1..gamma)
    uint32_t slice_bytes;
    int ring;               // streaming kernel: chunk slots per warp
    int seg_vectors;        // streaming kernel: 16-byte vectors per warp segment
    float *loss;            // [N]
    float *alpha;           // [N, gamma] or null
    float *grad;            // [N, gamma, V]
    int32_t *flags;         // [N] or null
    int shared_target;      // 1: target is [N + gamma - 1, V], pair (t, k) on row t + k
    int loss_kind;          // 0: e2e loss; 1: sum_k clamp(1 - alpha_k, 0, tau_max)
    float tau_max;
    const int32_t *topk_idx;  // top-K mode: [N, gamma, K] vocabulary indices (target = [N, gamma, K] values)
    int K;
    int grad32;             // the gradient base is 32-byte aligned: bf16 rows store 32 bytes at once
    // fault injection (TMEM-resident TV kernel; tests of the bounded waits)
    uint32_t wait_ns;       // limit of every on-chip wait; 0 = 2 s
    int skip_t;             // the position whose first exchange push warp 0 of CTA 0 skips; -1 = none
};

// Modes of the streaming row-pair statistics kernel.
enum PairMode { PAIR_STATS = 0, PAIR_DIAG = 1 };

struct PairArgs {
    const void *target;  // [B, gamma+1, V]
    const void *draft;   // [B, gamma, V]
    const float *temp;   // [B]
    int B, gamma, V;
    int ring;            // chunk slots per warp
    int seg_vectors;     // 16-byte vectors per warp segment
    float *alpha;        // [B, gamma] or null
    float *ent_p;        // [B, gamma+1] or null
    float *ent_q;        // [B, gamma] or null   (diagnostics)
    float *kl;           // [B, gamma] or null   (diagnostics)
    int32_t *yhat;       // [B, gamma] or null   (diagnostics)
    float *p_yhat;       // [B, gamma] or null   (diagnostics)
    int32_t *rs_better;  // [B, gamma] or null   (diagnostics)
    int32_t *flags;      // [B] or null
};

// Shared-memory header bytes in front of the slice buffers of each kernel.
uint32_t row_hdr_bytes();
uint32_t tv_hdr_bytes();
// Threads per CTA of each kernel.
int row_threads();
int tv_threads();

// Streaming verify kernel geometry.
uint32_t stream_hdr_bytes();
uint32_t stream_rec_bytes(int gamma, int S);
int stream_max_gamma();
int stream_threads();
uint32_t stream_slot_bytes(int cv);
int stream_max_chunks();
int stream_max_segments();
int stream_max_ring();

// Kernel entry points (host-side function pointers for cudaLaunchKernelEx).
const void *row_kernel(int dtype, int mode);
// cv: 128, 160 or 192 vectors per chunk; mode 0 = rejection sampling, 1 = target-only,
// 2 = rejection sampling with the Gumbel-max final draw; dbl: every sequence is a
// single target row (draft sampling), two chunks of it per ring slot (mode 0 at
// cv 160; other shapes ignore it)
const void *stream_kernel(int dtype, int cv, int mode, bool dbl = false);
const void *tv_kernel(int dtype);
// streaming TV kernel, cv: 128, 160 or 192; topk: the target is K cached entries per pair
const void *tvs_kernel(int dtype, int cv, bool topk = false);
// Streaming row-pair statistics kernel (mode: PairMode), cv: 128, 160 or 192.
const void *pair_kernel(int dtype, int cv, int mode);
uint32_t pair_hdr_bytes();
uint32_t pair_rec_bytes(int gamma, int S, int mode);
int pair_threads();
int pair_max_gamma();
int pair_max_segments();
int pair_max_ring();

// TMEM-resident TV kernel: the draft rows of a position parked in tensor
// memory.  ns: 16-byte vectors per lane and row (2, 4, 5, 8 or 10); null for
// another.
const void *tvm_kernel(int dtype, int ns);
uint32_t tvm_smem_bytes(int gamma, int C, int ns, int ring);
int tvm_threads();
int tvm_max_gamma();
int tvm_max_ring();
int tvm_warp_cols();
int tvm_max_cluster();
int tvm_team_warps();  // warps of one team per CTA (segments per CTA of a position)
int tvm_teams();       // independent teams per CTA

// TMEM-resident row-statistics kernel: draft rows parked in tensor memory
// for the overlap pass.  ns: 16-byte vectors per lane and row (2, 4, 5, 8,
// 10 or 15); null for another.
const void *stm_kernel(int dtype, int ns);
uint32_t stm_smem_bytes(int gamma, int C, int ns, int ring);
int stm_threads();
int stm_max_gamma();
int stm_max_ring();
int stm_warp_cols();
int stm_max_cluster();
int stm_parked();  // draft rows parked at a time

// Streaming TV kernel geometry.
uint32_t tvs_hdr_bytes();
uint32_t tvs_rec_bytes(int gamma, int S);
uint32_t tvs_bits_bytes(int gamma, int nvs);
int tvs_threads();
int tvs_max_gamma();
int tvs_max_segments();

}  // namespace mtp
