// api.cu -- the C ABI of libdflv (declared in include/dflv.h): host-side
// validation of shapes and pointers, then one asynchronous launch sequence on
// the caller's stream.  No allocation, no synchronisation, no global state.
#include <cstdint>

#include "../../include/dflv.h"
#include "kernels.h"

namespace {

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool aligned4(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }

dflv_status from_cuda(cudaError_t e) { return e == cudaSuccess ? DFLV_OK : DFLV_ERR_CUDA; }

dflv_status check_gdn_desc(const dflv_gdn_desc* d) {
    if (!d) return DFLV_ERR_INVALID_ARG;
    if (d->B < 1 || d->N_max < 1 || d->Hk < 1 || d->Hv < 1 || d->dk < 1 || d->dv < 1)
        return DFLV_ERR_INVALID_ARG;
    if (d->Hv % d->Hk != 0) return DFLV_ERR_INVALID_ARG;
    if (d->flags & ~(uint32_t)DFLV_FLAG_EARLY_PREFETCH) return DFLV_ERR_INVALID_ARG;
    if (d->N_max > 64) return DFLV_ERR_UNSUPPORTED;
    if (d->dk != 16 && d->dk != 32 && d->dk != 64 && d->dk != 128) return DFLV_ERR_UNSUPPORTED;
    if (d->dv % 16 != 0 || d->dv > 512) return DFLV_ERR_UNSUPPORTED;
    return DFLV_OK;
}

dflv_status check_attn_desc(const dflv_attn_desc* d) {
    if (!d) return DFLV_ERR_INVALID_ARG;
    if (d->B < 1 || d->N_max < 1 || d->Hq < 1 || d->Hkv < 1 || d->D < 1 || d->cap < 1 || d->window < 0)
        return DFLV_ERR_INVALID_ARG;
    if (d->Hq % d->Hkv != 0) return DFLV_ERR_INVALID_ARG;
    if (d->flags & ~(uint32_t)DFLV_FLAG_EARLY_PREFETCH) return DFLV_ERR_INVALID_ARG;
    if (d->N_max > 64) return DFLV_ERR_UNSUPPORTED;
    if (d->cap < d->N_max) return DFLV_ERR_CAPACITY;
    if (!(d->scale == d->scale)) return DFLV_ERR_INVALID_ARG;
    switch (d->type) {
        case DFLV_KV_Q8_0:
        case DFLV_KV_Q4_0:
            if (d->D != 64 && d->D != 128 && d->D != 256) return DFLV_ERR_UNSUPPORTED;
            break;
        case DFLV_KV_F32:
            if (d->D % 4 != 0 || d->D > 256) return DFLV_ERR_UNSUPPORTED;
            break;
        case DFLV_KV_Q8_0_Q4_0:
        case DFLV_KV_Q4_0_Q8_0:
        case DFLV_KV_TQ3_0:
            if (d->D != 128 && d->D != 256) return DFLV_ERR_UNSUPPORTED;
            break;
        default:
            return DFLV_ERR_UNSUPPORTED;
    }
    return DFLV_OK;
}

dflv_status check_kv_layer(const dflv_attn_desc* d, const dflv_kv_layer* c) {
    if (!c || !c->kq || !c->vq || !aligned16(c->kq) || !aligned16(c->vq)) return DFLV_ERR_INVALID_ARG;
    if (d->type != DFLV_KV_F32) {
        // the scale planes are read by the bulk-copy engine from 16-byte
        // aligned addresses
        if (!c->ks || !c->vs || !aligned16(c->ks) || !aligned16(c->vs)) return DFLV_ERR_INVALID_ARG;
    }
    return DFLV_OK;
}

dflv_status fill_gdn_args(const dflv_gdn_desc* desc, const int32_t* parent, const int32_t* n_nodes,
                          const uint16_t* q, const uint16_t* k, const uint16_t* v, const float* beta,
                          const float* log_alpha, const float* state, float* out, const dflv_gdn_factors* factors,
                          int32_t* status_dev, dflv::GdnVerifyArgs& a) {
    dflv_status s = check_gdn_desc(desc);
    if (s != DFLV_OK) return s;
    if (!parent || !n_nodes || !q || !k || !v || !beta || !log_alpha || !state || !out || !factors ||
        !factors->u || !factors->g || !factors->kcopy || !status_dev)
        return DFLV_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(state) || !aligned16(factors->kcopy) ||
        !aligned4(parent) || !aligned4(n_nodes) || !aligned4(beta) || !aligned4(log_alpha) ||
        !aligned4(out) || !aligned4(factors->u) || !aligned4(factors->g) || !aligned4(status_dev))
        return DFLV_ERR_INVALID_ARG;
    a.B = desc->B;
    a.N_max = desc->N_max;
    a.Hk = desc->Hk;
    a.Hv = desc->Hv;
    a.dk = desc->dk;
    a.dv = desc->dv;
    a.flags = desc->flags;
    a.parent = parent;
    a.n_nodes = n_nodes;
    a.q = q;
    a.k = k;
    a.v = v;
    a.beta = beta;
    a.log_alpha = log_alpha;
    a.state = state;
    a.out = out;
    a.u = factors->u;
    a.g = factors->g;
    a.kcopy = factors->kcopy;
    a.status = status_dev;
    return DFLV_OK;
}

dflv_status check_conv_desc(const dflv_conv_desc* d) {
    if (!d) return DFLV_ERR_INVALID_ARG;
    if (d->B < 1 || d->N_max < 1 || d->C < 1 || d->K < 1) return DFLV_ERR_INVALID_ARG;
    if (d->flags & ~(uint32_t)DFLV_FLAG_EARLY_PREFETCH) return DFLV_ERR_INVALID_ARG;
    if (d->N_max > 64 || d->K < 2 || d->K > 8 || d->C % 4 != 0) return DFLV_ERR_UNSUPPORTED;
    return DFLV_OK;
}

}  // namespace

extern "C" {

const char* dflv_status_string(dflv_status s) {
    switch (s) {
        case DFLV_OK: return "ok";
        case DFLV_ERR_INVALID_ARG: return "invalid argument (null or misaligned pointer, bad count)";
        case DFLV_ERR_TOPOLOGY: return "invalid tree topology";
        case DFLV_ERR_UNSUPPORTED: return "unsupported shape or type";
        case DFLV_ERR_CAPACITY: return "capacity exceeded";
        case DFLV_ERR_CUDA: return "CUDA launch error";
    }
    return "unknown status";
}

size_t dflv_gdn_workspace_size(const dflv_gdn_desc*) { return 0; }
size_t dflv_attn_workspace_size(const dflv_attn_desc* desc) {
    if (check_attn_desc(desc) != DFLV_OK) return 0;
    dflv::AttnVerifyArgs a = {};
    a.B = desc->B;
    a.N_max = desc->N_max;
    a.Hq = desc->Hq;
    a.Hkv = desc->Hkv;
    a.D = desc->D;
    a.cap = desc->cap;
    a.window = desc->window;
    a.type = desc->type;
    return dflv::attn_workspace_bytes(a);
}

dflv_status dflv_tree_gdn_verify(const dflv_gdn_desc* desc, const int32_t* parent,
                                 const int32_t* n_nodes, const uint16_t* q, const uint16_t* k,
                                 const uint16_t* v, const float* beta, const float* log_alpha,
                                 const float* state, float* out, const dflv_gdn_factors* factors,
                                 int32_t* status_dev, void* workspace, size_t ws_bytes,
                                 dflv_stream_t stream) {
    (void)workspace;
    (void)ws_bytes;
    dflv::GdnVerifyArgs a = {};
    dflv_status s = fill_gdn_args(desc, parent, n_nodes, q, k, v, beta, log_alpha, state, out, factors,
                                  status_dev, a);
    if (s != DFLV_OK) return s;
    return from_cuda(dflv::launch_gdn_tree_verify(a, reinterpret_cast<cudaStream_t>(stream)));
}

dflv_status dflv_tree_gdn_verify_pending(const dflv_gdn_desc* desc, const int32_t* parent,
                                         const int32_t* n_nodes, const uint16_t* q, const uint16_t* k,
                                         const uint16_t* v, const float* beta, const float* log_alpha,
                                         float* state, const dflv_gdn_factors* pending,
                                         const int32_t* pending_path, const int32_t* pending_len,
                                         float* out, const dflv_gdn_factors* factors,
                                         int32_t* status_dev, void* workspace, size_t ws_bytes,
                                         dflv_stream_t stream) {
    (void)workspace;
    (void)ws_bytes;
    dflv::GdnVerifyArgs a = {};
    dflv_status s = fill_gdn_args(desc, parent, n_nodes, q, k, v, beta, log_alpha, state, out, factors,
                                  status_dev, a);
    if (s != DFLV_OK) return s;
    if (!pending || !pending->u || !pending->g || !pending->kcopy || !pending_path || !pending_len)
        return DFLV_ERR_INVALID_ARG;
    if (!aligned16(pending->u) || !aligned16(pending->kcopy) || !aligned4(pending->g) || !aligned4(pending_path) ||
        !aligned4(pending_len))
        return DFLV_ERR_INVALID_ARG;
    if (pending->u == factors->u || pending->g == factors->g || pending->kcopy == factors->kcopy)
        return DFLV_ERR_INVALID_ARG;  // the new factors would overwrite the pending ones
    a.pend_u = pending->u;
    a.pend_g = pending->g;
    a.pend_k = pending->kcopy;
    a.pend_path = pending_path;
    a.pend_len = pending_len;
    a.state_out = state;
    return from_cuda(dflv::launch_gdn_tree_verify(a, reinterpret_cast<cudaStream_t>(stream)));
}

dflv_status dflv_tree_attn_verify(const dflv_attn_desc* desc, const int32_t* parent,
                                  const int32_t* n_nodes, const int32_t* n_past,
                                  const uint16_t* q, const uint16_t* k_new,
                                  const uint16_t* v_new, const dflv_kv_layer* cache, float* out,
                                  int32_t* status_dev, void* workspace, size_t ws_bytes,
                                  dflv_stream_t stream) {
    dflv_status s = check_attn_desc(desc);
    if (s != DFLV_OK) return s;
    if (!parent || !n_nodes || !n_past || !q || !k_new || !v_new || !out || !status_dev)
        return DFLV_ERR_INVALID_ARG;
    s = check_kv_layer(desc, cache);
    if (s != DFLV_OK) return s;
    if (!aligned16(q) || !aligned16(k_new) || !aligned16(v_new) || !aligned16(out) || !aligned4(parent) ||
        !aligned4(n_nodes) || !aligned4(n_past) || !aligned4(status_dev) || (workspace && !aligned16(workspace)))
        return DFLV_ERR_INVALID_ARG;
    dflv::AttnVerifyArgs a = {};
    a.B = desc->B;
    a.N_max = desc->N_max;
    a.Hq = desc->Hq;
    a.Hkv = desc->Hkv;
    a.D = desc->D;
    a.cap = desc->cap;
    a.window = desc->window;
    a.type = desc->type;
    a.scale = desc->scale;
    a.flags = desc->flags;
    a.parent = parent;
    a.n_nodes = n_nodes;
    a.n_past = n_past;
    a.q = q;
    a.k_new = k_new;
    a.v_new = v_new;
    a.kq = cache->kq;
    a.vq = cache->vq;
    a.ks = cache->ks;
    a.vs = cache->vs;
    a.out = out;
    a.status = status_dev;
    a.ws = workspace;
    a.ws_bytes = workspace ? ws_bytes : 0;
    return from_cuda(dflv::launch_attn_tree_verify(a, reinterpret_cast<cudaStream_t>(stream)));
}

dflv_status dflv_accept_greedy(int32_t B, int32_t N_max, int32_t vocab, const float* logits,
                               const int32_t* tokens, const int32_t* parent,
                               const int32_t* n_nodes, int32_t* path, int32_t* path_len,
                               int32_t* next_token, int32_t* best, int32_t* status_dev,
                               dflv_stream_t stream) {
    if (B < 1 || N_max < 1 || vocab < 1) return DFLV_ERR_INVALID_ARG;
    if (N_max > 64) return DFLV_ERR_UNSUPPORTED;
    if (!logits || !tokens || !parent || !n_nodes || !path || !path_len || !next_token || !best ||
        !status_dev)
        return DFLV_ERR_INVALID_ARG;
    if (!aligned16(logits) || !aligned4(tokens) || !aligned4(parent) || !aligned4(n_nodes) ||
        !aligned4(path) || !aligned4(path_len) || !aligned4(next_token) || !aligned4(best) ||
        !aligned4(status_dev))
        return DFLV_ERR_INVALID_ARG;
    dflv::AcceptArgs a;
    a.B = B;
    a.N_max = N_max;
    a.vocab = vocab;
    a.logits = logits;
    a.tokens = tokens;
    a.parent = parent;
    a.n_nodes = n_nodes;
    a.path = path;
    a.path_len = path_len;
    a.next_token = next_token;
    a.best = best;
    a.status = status_dev;
    return from_cuda(dflv::launch_accept_greedy(a, reinterpret_cast<cudaStream_t>(stream)));
}

dflv_status dflv_commit_rollback(const dflv_gdn_desc* gdn, int32_t n_gdn, float* const* states,
                                 const dflv_gdn_factors* factors, const dflv_attn_desc* attn,
                                 int32_t n_attn, const dflv_kv_layer* caches,
                                 const int32_t* path, const int32_t* path_len, int32_t* n_past,
                                 int32_t* status_dev, dflv_stream_t stream) {
    if (n_gdn < 0 || n_attn < 0) return DFLV_ERR_INVALID_ARG;
    if (n_gdn > DFLV_MAX_COMMIT_GDN_LAYERS || n_attn > DFLV_MAX_COMMIT_ATTN_LAYERS)
        return DFLV_ERR_UNSUPPORTED;
    if (!path || !path_len || !status_dev || !aligned4(path) || !aligned4(path_len) || !aligned4(status_dev))
        return DFLV_ERR_INVALID_ARG;
    dflv::CommitArgs a = {};
    a.n_gdn = n_gdn;
    a.n_attn = n_attn;
    a.path = path;
    a.path_len = path_len;
    a.n_past = n_past;
    a.status = status_dev;
    int B = -1, N_max = -1;
    if (n_gdn > 0) {
        dflv_status s = check_gdn_desc(gdn);
        if (s != DFLV_OK) return s;
        if (!states || !factors) return DFLV_ERR_INVALID_ARG;
        if (gdn->dk % 4 != 0) return DFLV_ERR_UNSUPPORTED;
        B = gdn->B;
        N_max = gdn->N_max;
        a.Hk = gdn->Hk;
        a.Hv = gdn->Hv;
        a.dk = gdn->dk;
        a.dv = gdn->dv;
        for (int l = 0; l < n_gdn; ++l) {
            if (!states[l] || !factors[l].u || !factors[l].g || !factors[l].kcopy || !aligned16(states[l]))
                return DFLV_ERR_INVALID_ARG;
            a.gdn[l].state = states[l];
            a.gdn[l].u = factors[l].u;
            a.gdn[l].g = factors[l].g;
            a.gdn[l].kcopy = factors[l].kcopy;
        }
    }
    if (n_attn > 0) {
        dflv_status s = check_attn_desc(attn);
        if (s != DFLV_OK) return s;
        if (!caches || !n_past) return DFLV_ERR_INVALID_ARG;
        if (B >= 0 && (attn->B != B || attn->N_max != N_max)) return DFLV_ERR_INVALID_ARG;
        B = attn->B;
        N_max = attn->N_max;
        a.Hkv = attn->Hkv;
        a.D = attn->D;
        a.cap = attn->cap;
        a.type = attn->type;
        for (int l = 0; l < n_attn; ++l) {
            s = check_kv_layer(attn, &caches[l]);
            if (s != DFLV_OK) return s;
            a.attn[l].kq = static_cast<uint8_t*>(caches[l].kq);
            a.attn[l].vq = static_cast<uint8_t*>(caches[l].vq);
            a.attn[l].ks = caches[l].ks;
            a.attn[l].vs = caches[l].vs;
        }
    }
    if (B < 0) {
        // nothing to commit into; n_past still advances when given
        if (!n_past) return DFLV_OK;
        return DFLV_ERR_INVALID_ARG;
    }
    if (n_past && !aligned4(n_past)) return DFLV_ERR_INVALID_ARG;
    a.B = B;
    a.N_max = N_max;
    return from_cuda(dflv::launch_commit_rollback(a, reinterpret_cast<cudaStream_t>(stream)));
}

}  // extern "C"

extern "C" {

dflv_status dflv_tree_conv_verify(const dflv_conv_desc* desc, const int32_t* parent,
                                  const int32_t* n_nodes, const uint16_t* x,
                                  const uint16_t* conv_state, const float* weight, float* out,
                                  int32_t* status_dev, dflv_stream_t stream) {
    dflv_status s = check_conv_desc(desc);
    if (s != DFLV_OK) return s;
    if (!parent || !n_nodes || !x || !conv_state || !weight || !out || !status_dev) return DFLV_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(conv_state) || !aligned16(weight) || !aligned16(out) || !aligned4(parent) ||
        !aligned4(n_nodes) || !aligned4(status_dev))
        return DFLV_ERR_INVALID_ARG;
    dflv::ConvVerifyArgs a;
    a.B = desc->B;
    a.N_max = desc->N_max;
    a.C = desc->C;
    a.K = desc->K;
    a.flags = desc->flags;
    a.parent = parent;
    a.n_nodes = n_nodes;
    a.x = x;
    a.state = conv_state;
    a.w = weight;
    a.out = out;
    a.status = status_dev;
    return from_cuda(dflv::launch_conv_tree_verify(a, reinterpret_cast<cudaStream_t>(stream)));
}

dflv_status dflv_conv_commit(const dflv_conv_desc* desc, int32_t n_layers, uint16_t* const* states,
                             const uint16_t* const* xs, const int32_t* path,
                             const int32_t* path_len, int32_t* status_dev, dflv_stream_t stream) {
    dflv_status s = check_conv_desc(desc);
    if (s != DFLV_OK) return s;
    if (n_layers < 1 || n_layers > DFLV_MAX_CONV_LAYERS || !states || !xs || !path || !path_len || !status_dev)
        return DFLV_ERR_INVALID_ARG;
    if (!aligned4(path) || !aligned4(path_len) || !aligned4(status_dev)) return DFLV_ERR_INVALID_ARG;
    static_assert(DFLV_MAX_CONV_LAYERS == dflv::kMaxConvLayers, "layer limits differ");
    dflv::ConvCommitArgs a = {};
    a.B = desc->B;
    a.N_max = desc->N_max;
    a.C = desc->C;
    a.K = desc->K;
    a.n_layers = n_layers;
    a.path = path;
    a.path_len = path_len;
    a.status = status_dev;
    for (int l = 0; l < n_layers; ++l) {
        if (!states[l] || !xs[l] || !aligned16(states[l]) || !aligned16(xs[l])) return DFLV_ERR_INVALID_ARG;
        a.state[l] = states[l];
        a.x[l] = xs[l];
    }
    return from_cuda(dflv::launch_conv_commit(a, reinterpret_cast<cudaStream_t>(stream)));
}

}  // extern "C"

extern "C" {

dflv_status dflv_ddtree_build(const dflv_ddtree_desc* desc, const float* draft_logits,
                              const int32_t* root_token, int32_t* topk_tok, float* topk_logp,
                              int32_t* parent, int32_t* tokens, int32_t* n_nodes, float* score,
                              int32_t* status_dev, dflv_stream_t stream) {
    if (!desc) return DFLV_ERR_INVALID_ARG;
    if (desc->B < 1 || desc->D < 1 || desc->K < 1 || desc->budget < 1 || desc->V < 1 || desc->flags != 0 ||
        desc->tau != desc->tau)
        return DFLV_ERR_INVALID_ARG;
    if (desc->D > dflv::kMaxTreeDepth || desc->K > 8 || desc->budget > 64 || desc->V % 4 != 0 || desc->V < desc->K)
        return DFLV_ERR_UNSUPPORTED;
    if (!draft_logits || !root_token || !topk_tok || !topk_logp || !parent || !tokens || !n_nodes || !score ||
        !status_dev)
        return DFLV_ERR_INVALID_ARG;
    if (!aligned16(draft_logits) || !aligned4(root_token) || !aligned4(topk_tok) || !aligned4(topk_logp) ||
        !aligned4(parent) || !aligned4(tokens) || !aligned4(n_nodes) || !aligned4(score) || !aligned4(status_dev))
        return DFLV_ERR_INVALID_ARG;
    dflv::DdtreeArgs a;
    a.B = desc->B;
    a.D = desc->D;
    a.V = desc->V;
    a.K = desc->K;
    a.budget = desc->budget;
    a.tau = desc->tau;
    a.logits = draft_logits;
    a.root_token = root_token;
    a.topk_tok = topk_tok;
    a.topk_logp = topk_logp;
    a.parent = parent;
    a.tokens = tokens;
    a.n_nodes = n_nodes;
    a.score = score;
    a.status = status_dev;
    return from_cuda(dflv::launch_ddtree_build(a, reinterpret_cast<cudaStream_t>(stream)));
}

}  // extern "C"
