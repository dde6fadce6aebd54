// kernels.h -- internal launch interface between the C ABI (api.cu) and the
// kernels.  Plain structs of device pointers and sizes; no torch types.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "../../include/dflv.h"

namespace dflv {

// Set by a verify launcher, never by a caller (the C ABI accepts only
// DFLV_FLAG_* bits): with early prefetch, and when every CTA of the launch
// can be resident at once (so that they all start under the preceding
// kernel), the kernel asks for its layer inputs in the L2 before its
// dependency wait.
constexpr unsigned kFlagPrefetchInputs = 1u << 16;

struct GdnVerifyArgs {
    int B, N_max, Hk, Hv, dk, dv;
    unsigned flags;  // DFLV_FLAG_*
    const int32_t* parent;
    const int32_t* n_nodes;
    const uint16_t* q;
    const uint16_t* k;
    const uint16_t* v;
    const float* beta;
    const float* log_alpha;
    const float* state;
    float* out;
    float* u;
    float* g;
    uint16_t* kcopy;
    int32_t* status;
    // deferred commit (null pointers: none): the previous verify's factors
    // and accepted path; the updated state rows are written to state_out
    const float* pend_u;
    const float* pend_g;
    const uint16_t* pend_k;
    const int32_t* pend_path;
    const int32_t* pend_len;
    float* state_out;
};

cudaError_t launch_gdn_tree_verify(const GdnVerifyArgs& a, cudaStream_t stream);
size_t gdn_verify_smem_bytes(int N_max, int dk, int dv);

struct AttnVerifyArgs {
    int B, N_max, Hq, Hkv, D, cap, window, type;
    float scale;
    unsigned flags;  // DFLV_FLAG_*
    const int32_t* parent;
    const int32_t* n_nodes;
    const int32_t* n_past;
    const uint16_t* q;
    const uint16_t* k_new;
    const uint16_t* v_new;
    void* kq;
    void* vq;
    uint16_t* ks;
    uint16_t* vs;
    float* out;
    int32_t* status;
    // caller's workspace (may be null): when it holds at least
    // attn_workspace_bytes(), the key splits merge through it
    void* ws;
    size_t ws_bytes;
};

cudaError_t launch_attn_tree_verify(const AttnVerifyArgs& a, cudaStream_t stream);
cudaError_t launch_attn_tree_verify_tc(const AttnVerifyArgs& a, cudaStream_t stream);
// Bytes of workspace with which a call of this shape merges its key splits
// through global memory (0: the shape never uses one).  Depends on the
// current device (the launch plan follows its cluster occupancy).
size_t attn_workspace_bytes(const AttnVerifyArgs& a);
size_t attn_workspace_bytes_tc(const AttnVerifyArgs& a);

// Code bytes of one cache row of plane `plane` (0: keys, 1: values) for a
// dflv_kv_type (the asymmetric types differ between the planes).
__host__ __device__ inline int kv_code_bytes(int type, int plane, int D) {
    int t = type;
    if (type == DFLV_KV_Q8_0_Q4_0) t = plane ? DFLV_KV_Q4_0 : DFLV_KV_Q8_0;
    else if (type == DFLV_KV_Q4_0_Q8_0) t = plane ? DFLV_KV_Q8_0 : DFLV_KV_Q4_0;
    return t == DFLV_KV_Q8_0 ? D : t == DFLV_KV_Q4_0 ? D / 2 : t == DFLV_KV_TQ3_0 ? D / 32 * 12 : D * 4;
}

struct AcceptArgs {
    int B, N_max, vocab;
    const float* logits;
    const int32_t* tokens;
    const int32_t* parent;
    const int32_t* n_nodes;
    int32_t* path;
    int32_t* path_len;
    int32_t* next_token;
    int32_t* best;
    int32_t* status;
};

cudaError_t launch_accept_greedy(const AcceptArgs& a, cudaStream_t stream);

constexpr int kMaxCommitGdn = 128;
constexpr int kMaxCommitAttn = 64;

struct CommitGdnLayer {
    float* state;
    const float* u;
    const float* g;
    const uint16_t* kcopy;
};

struct CommitAttnLayer {
    uint8_t* kq;
    uint8_t* vq;
    uint16_t* ks;
    uint16_t* vs;
};

// Passed by value as a kernel parameter (a few KB; graph-capturable).
struct CommitArgs {
    int B, N_max;
    // GDN geometry
    int n_gdn, Hk, Hv, dk, dv;
    // attention geometry
    int n_attn, Hkv, D, cap, type;
    const int32_t* path;
    const int32_t* path_len;
    int32_t* n_past;
    int32_t* status;
    CommitGdnLayer gdn[kMaxCommitGdn];
    CommitAttnLayer attn[kMaxCommitAttn];
};

cudaError_t launch_commit_rollback(const CommitArgs& a, cudaStream_t stream);

struct ConvVerifyArgs {
    int B, N_max, C, K;
    unsigned flags;  // DFLV_FLAG_*
    const int32_t* parent;
    const int32_t* n_nodes;
    const uint16_t* x;
    const uint16_t* state;
    const float* w;
    float* out;
    int32_t* status;
};

cudaError_t launch_conv_tree_verify(const ConvVerifyArgs& a, cudaStream_t stream);

constexpr int kMaxConvLayers = 128;

// Passed by value as a kernel parameter (2 KB of pointers).
struct ConvCommitArgs {
    int B, N_max, C, K, n_layers;
    const int32_t* path;
    const int32_t* path_len;
    int32_t* status;
    uint16_t* state[kMaxConvLayers];
    const uint16_t* x[kMaxConvLayers];
};

cudaError_t launch_conv_commit(const ConvCommitArgs& a, cudaStream_t stream);

constexpr int kMaxTreeDepth = 64;

struct DdtreeArgs {
    int B, D, V, K, budget;
    float tau;  // < 0: no pruning
    const float* logits;
    const int32_t* root_token;
    int32_t* topk_tok;
    float* topk_logp;
    int32_t* parent;
    int32_t* tokens;
    int32_t* n_nodes;
    float* score;
    int32_t* status;
};

cudaError_t launch_ddtree_build(const DdtreeArgs& a, cudaStream_t stream);

}  // namespace dflv
