/*
 * dflv.h -- C ABI of libdflv, the GPU tree-verify step of DDTree speculative
 * decoding for a hybrid gated-DeltaNet + full-attention target.
 *
 * Sources for what the step computes (the pages this library follows):
 *   [README]  "Luce DFlash" server README (Luce-Org/lucebox, server/README.md)
 *   [PR606]   lucebox PR #606 "add SpecLA factor-capture speculative decoding"
 *
 *   - A draft tree of n nodes is given as candidate tokens plus a parent
 *     array in topological order; node 0 is the root (the last committed
 *     token) and parent[i] < i.  One target pass scores every node, with a
 *     causal mask derived from the parent pointers ([README] "How it works",
 *     "DDTree tree verify"; [PR606] "Paper mapping": scored candidates and
 *     parent topology, a chain being a degenerate tree).
 *   - In the gated-DeltaNet layers each node's recurrent state is its
 *     parent's state advanced by one gated delta-rule step ([README]
 *     "Architecture note": ggml_gated_delta_net_tree).  The pages do not
 *     write the recurrence; this library uses the standard gated delta rule
 *         S_i = alpha_i S_par(i) (I - beta_i k_i k_i^T) + beta_i v_i k_i^T,
 *         o_i = S_i q_i,
 *     with the committed state as the root's parent state, q and k given
 *     already L2-normalised, and no 1/sqrt(dk) factor.
 *   - In the attention layers the tree queries attend to the block-quantised
 *     KV cache and to their own ancestors-or-self, optionally inside a
 *     sliding window ([README] "--fa-window N", 0 = full attention;
 *     "Asymmetric K/V quantization": q8_0 default, Q4_0 at 4.5 bpv).
 *   - Greedy acceptance walks the tree against the target's argmax ([README]
 *     "Scope and limits": the DDTree verify skeleton stays argmax).
 *   - Commit / rollback leaves the recurrent state and KV cache as if only
 *     the accepted path had been decoded ([README] "How it works",
 *     "Per-step rollback"; [PR606] review note naming the commit routines).
 *   - The draft tree itself is built best-first over the draft's top-K
 *     tokens per position after a rank-0 chain ([README] "How it works").
 *   - The short convolution in front of each gated-DeltaNet layer reads
 *     each node's window along its parent chain ([README] "How it works":
 *     ggml_ssm_conv_tree).
 *
 * General conventions
 *   - Every array argument is a DEVICE pointer unless marked "host".  The
 *     caller owns every buffer; the library never allocates or frees memory
 *     (dflv_tree_attn_verify_noalloc uses one fixed scratch array of the
 *     library's own instead, below).
 *   - bf16 and fp16 values are passed as uint16_t bit patterns.
 *   - All calls are asynchronous on the given stream (0 = legacy default
 *     stream) and never synchronise it, so a whole step can be captured in a
 *     CUDA graph.
 *   - The returned dflv_status reports only what the host can check before
 *     launching (NULL or misaligned pointers, unsupported shapes).  Nothing
 *     is launched when it is not DFLV_OK.
 *   - Errors found on the device (a malformed parent array, a cache slot out
 *     of capacity, an invalid accepted path) are OR-ed into *status_dev as
 *     DFLV_DEV_* bits; the outputs of the affected sequence are then
 *     unspecified.  status_dev points to one int32 in device memory that the
 *     caller zeroes and reads back when it wants to check.
 *   - Pointers to bf16/f32/int8/u8 arrays and to the fp16 scale planes of a
 *     KV cache must be 16-byte aligned.
 *   - No global state: calls are re-entrant on distinct buffers (except
 *     dflv_tree_attn_verify_noalloc, whose calls on one device share its
 *     scratch array).
 *   - Padded nodes (i >= n_nodes[b]) are ignored; their outputs are
 *     unspecified.
 */
#ifndef DFLV_H
#define DFLV_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* dflv_stream_t; /* a cudaStream_t */

typedef enum {
    DFLV_OK = 0,
    DFLV_ERR_INVALID_ARG = 1, /* NULL / misaligned pointer, bad count */
    DFLV_ERR_TOPOLOGY = 2,    /* reserved for host-visible topology errors */
    DFLV_ERR_UNSUPPORTED = 3, /* shape or type this build does not implement */
    DFLV_ERR_CAPACITY = 4,    /* a workspace or cache too small (host check) */
    DFLV_ERR_CUDA = 5         /* a CUDA launch or attribute call failed */
} dflv_status;

/* Bits OR-ed into *status_dev by the kernels. */
enum {
    DFLV_DEV_TOPOLOGY = 1, /* parent[0] != -1, parent[i] outside [0, i), n outside [1, N_max] */
    DFLV_DEV_CAPACITY = 2, /* P < 0 or P + n > cap in an attention layer */
    DFLV_DEV_PATH = 4,     /* an accepted path with a length outside the call's range (each call
                              states it) or a node outside [0, N_max) */
    DFLV_DEV_TIMEOUT = 8   /* a bounded wait for an asynchronous copy gave up */
};

typedef enum {
    DFLV_KV_Q8_0 = 0, /* 32 int8 codes + one fp16 scale d per block: x = d * q */
    DFLV_KV_Q4_0 = 1, /* 32 4-bit codes c + one fp16 scale d per block: x = d * (c - 8) */
    DFLV_KV_F32 = 2,  /* plain fp32 cache (small exactness checks) */
    /* Asymmetric caches ([README] "Asymmetric K/V quantization": keys and
     * values quantised independently), head sizes 128 and 256: */
    DFLV_KV_Q8_0_Q4_0 = 3, /* keys q8_0, values q4_0 */
    DFLV_KV_Q4_0_Q8_0 = 4, /* keys q4_0, values q8_0 */
    /* TQ3_0 ([README] "Results" KV note: TQ3_0 at 3.5 bits per value, the
     * default; "Asymmetric K/V quantization": a fast Walsh-Hadamard rotation
     * applied to the query and undone on the attention output when the keys
     * are TQ3_0).  Keys and values both: each cached row is the orthonormal
     * Walsh-Hadamard transform (Sylvester order, over the whole head) of the
     * bf16 row, in blocks of 32 with one fp16 scale d = amax / 3 and 32
     * three-bit codes c = clamp(round-half-away(x * (1/d)), -4, 3) + 4, code j
     * in bits 3j .. 3j+2 of the block's 12 little-endian bytes; x = d * (c - 4)
     * in the rotated basis.  Head sizes 128 and 256. */
    DFLV_KV_TQ3_0 = 5
} dflv_kv_type;

/* Launch overlap.  Every kernel of this library is launched with
 * programmatic dependent launch: it may be scheduled while the preceding
 * kernel on the stream finishes, and it waits for that kernel's completion
 * (and memory) before it reads anything.  With DFLV_FLAG_EARLY_PREFETCH in a
 * verify call's descriptor, the kernel starts reading the inputs that the
 * step itself never produces before that wait: for gated-DeltaNet the
 * committed state and the tree (parent, n_nodes), for attention the tree,
 * n_past and the cached slots below P.  Set the flag only when the kernel
 * that immediately precedes the call on the stream writes none of these
 * buffers -- in a verify step, every layer after the first.  (Each kernel
 * of the library releases its successor only after its own wait, so the
 * overlap never reaches past the immediate predecessor.)  Before its wait a
 * kernel may also ask for inputs the preceding kernel produces (a verify's
 * q, k, v, beta, log_alpha and new keys/values; the acceptance's logits) to
 * be brought into the L2, where a model's producing layer has just left
 * them; such a request moves no data into the kernel and orders nothing, so
 * the values it reads after the wait are the ones the predecessor wrote.
 * The verify kernels do so only with the flag set and when all their CTAs
 * fit on the device at once. */
enum { DFLV_FLAG_EARLY_PREFETCH = 1 };

/* ------------------------------------------------------------------------ */
/* Gated-DeltaNet layer                                                      */
/* ------------------------------------------------------------------------ */

/* Shape of one gated-DeltaNet layer's verify.  Hv must be a multiple of Hk;
 * v-head h reads q/k head h / (Hv / Hk).  Supported: 1 <= N_max <= 64,
 * dk in {16, 32, 64, 128}, dv a multiple of 16 (<= 512). */
typedef struct {
    int32_t B, N_max, Hk, Hv, dk, dv;
    uint32_t flags; /* 0 or DFLV_FLAG_EARLY_PREFETCH */
} dflv_gdn_desc;

/* Per-node factors captured by verify for commit ([PR606]: factor capture
 * instead of materialising every node's state; [README]: the _persist op
 * writes these intermediates directly instead of copying states).  All
 * caller-owned device arrays:
 *   u     [B][N_max][Hv][dv] f32 : u_i = beta_i (v_i - alpha_i S_par(i) k_i)
 *   g     [B][N_max][Hv]     f32 : g_i = sum of log alpha over i's ancestors-or-self
 *   kcopy [B][N_max][Hk][dk] bf16: the node keys (so the caller may reuse k)
 * Valid until the next verify that writes the same buffers. */
typedef struct {
    float* u;
    float* g;
    uint16_t* kcopy;
} dflv_gdn_factors;

/* Tree verify of one gated-DeltaNet layer.
 *   parent    [B][N_max] int32; n_nodes [B] int32
 *   q, k      [B][N_max][Hk][dk] bf16 (L2-normalised by the caller)
 *   v         [B][N_max][Hv][dv] bf16
 *   beta      [B][N_max][Hv] f32;  log_alpha [B][N_max][Hv] f32 (log of the decay)
 *   state     [B][Hv][dv][dk] f32, the committed state; READ ONLY here
 *   out       [B][N_max][Hv][dv] f32, o_i = S_i q_i
 *   factors   host pointer to the factor buffers above (all required)
 *   workspace reserved: dflv_gdn_workspace_size() returns 0; may be NULL
 * The committed state is never written, so rejecting the whole tree costs
 * nothing (rollback is free). */
dflv_status dflv_tree_gdn_verify(const dflv_gdn_desc* desc, const int32_t* parent,
                                 const int32_t* n_nodes, const uint16_t* q, const uint16_t* k,
                                 const uint16_t* v, const float* beta, const float* log_alpha,
                                 const float* state, float* out, const dflv_gdn_factors* factors,
                                 int32_t* status_dev, void* workspace, size_t ws_bytes,
                                 dflv_stream_t stream);

/* Deferred commit ([PR606]: SpecLA keeps the accepted path's factors pending
 * and applies them while the state streams into the next verify).  Tree
 * verify of one gated-DeltaNet layer whose committed state still owes the
 * previous step's accepted path:
 *   state        [B][Hv][dv][dk] f32, IN/OUT: on entry the state before the
 *                previous step's commit of this layer; every row is first
 *                brought up to date,
 *                  S <- e^{g_e} S + sum_{m<L} e^{g_e - g_{p_m}} u_{p_m} k_{p_m}^T
 *                (p_m = pending_path[b][m], e = p_{L-1}, u/g/kcopy from
 *                pending: the update dflv_commit_rollback applies), written
 *                back, and the tree is verified against the updated state.
 *   pending      the previous verify's factors of this layer (read only; must
 *                not alias `factors`, which receives this verify's factors)
 *   pending_path [B][N_max] int32, pending_len [B] int32: the previous step's
 *                accepted path (dflv_accept_greedy output); pending_len[b] = 0
 *                leaves sequence b's state as it is.  A length outside
 *                [0, N_max] or a node outside [0, N_max) raises
 *                DFLV_DEV_PATH and that sequence's update is skipped.
 * Everything else as dflv_tree_gdn_verify (same descriptor, N_max equal to
 * the previous verify's).  With DFLV_FLAG_EARLY_PREFETCH the tree, pending
 * factors and pending path are read, and the state rows are read, brought up
 * to date and written back, before the dependency wait: the kernel
 * immediately before the call must not write those buffers, nor read the
 * state.
 * A step then commits only the KV caches (dflv_commit_rollback with
 * n_gdn = 0); the final pending update of a sequence can be applied with
 * dflv_commit_rollback as usual. */
dflv_status dflv_tree_gdn_verify_pending(const dflv_gdn_desc* desc, const int32_t* parent,
                                         const int32_t* n_nodes, const uint16_t* q, const uint16_t* k,
                                         const uint16_t* v, const float* beta, const float* log_alpha,
                                         float* state, const dflv_gdn_factors* pending,
                                         const int32_t* pending_path, const int32_t* pending_len,
                                         float* out, const dflv_gdn_factors* factors,
                                         int32_t* status_dev, void* workspace, size_t ws_bytes,
                                         dflv_stream_t stream);

size_t dflv_gdn_workspace_size(const dflv_gdn_desc* desc);

/* ------------------------------------------------------------------------ */
/* Short convolution in front of a gated-DeltaNet layer                      */
/* ------------------------------------------------------------------------ */

/* The depthwise causal convolution of width K that feeds a gated-DeltaNet
 * layer, evaluated on the tree ([README] "How it works": ggml_ssm_conv_tree,
 * each node reads its K-1 window along the parent chain).  The pages name
 * the op but do not write it; this library computes, per channel c,
 *     out[b][i][c] = sum_{j<K} weight[c][j] * w_j,
 * where w_{K-1} is node i's own input, w_{K-2} its parent's, and so on up
 * the parent chain; once the chain has passed the root, w continues with
 * the conv state (the K-1 inputs before the root, newest last).  No bias and
 * no activation (the caller applies those).  A chain tree therefore gives
 * the sequential causal convolution.
 * Supported: 1 <= N_max <= 64, 2 <= K <= 8, C a multiple of 4. */
typedef struct {
    int32_t B, N_max, C, K;
    uint32_t flags; /* 0 or DFLV_FLAG_EARLY_PREFETCH */
} dflv_conv_desc;

/* Tree verify of one short-convolution layer.
 *   parent     [B][N_max] int32; n_nodes [B] int32
 *   x          [B][N_max][C] bf16: the nodes' inputs (the layer's q/k/v
 *              projections before the convolution)
 *   conv_state [B][K-1][C] bf16: the committed window, oldest first; READ
 *              ONLY here
 *   weight     [C][K] f32: tap K-1 multiplies the current node
 *   out        [B][N_max][C] f32; rows of padded nodes are not written
 * With DFLV_FLAG_EARLY_PREFETCH the tree, weight and conv_state are read
 * before the dependency wait (x after it).  A malformed tree raises
 * DFLV_DEV_TOPOLOGY and that sequence writes nothing. */
dflv_status dflv_tree_conv_verify(const dflv_conv_desc* desc, const int32_t* parent,
                                  const int32_t* n_nodes, const uint16_t* x,
                                  const uint16_t* conv_state, const float* weight, float* out,
                                  int32_t* status_dev, dflv_stream_t stream);

/* Commits the accepted path into the conv state of n_layers layers in one
 * launch: each state becomes the last K-1 entries of
 * [conv_state ; x of path[b][0..L)], the window that decoding only the
 * accepted tokens leaves behind ([README] "How it works", per-step rollback
 * of the recurrent state).
 *   states  host array of n_layers device pointers, [B][K-1][C] bf16 (in/out)
 *   xs      host array of n_layers device pointers, [B][N_max][C] bf16: the
 *           inputs that layer's verify read
 *   path, path_len  [B][N_max], [B] int32 (dflv_accept_greedy output);
 *           path_len[b] = 0 leaves sequence b unchanged; a length outside
 *           [0, N_max] or a node outside [0, N_max) raises DFLV_DEV_PATH
 *           and that sequence is left unchanged.
 * 1 <= n_layers <= DFLV_MAX_CONV_LAYERS.  All reads of a state precede its
 * writes (each thread owns its channels). */
dflv_status dflv_conv_commit(const dflv_conv_desc* desc, int32_t n_layers, uint16_t* const* states,
                             const uint16_t* const* xs, const int32_t* path,
                             const int32_t* path_len, int32_t* status_dev, dflv_stream_t stream);

#define DFLV_MAX_CONV_LAYERS 128

/* ------------------------------------------------------------------------ */
/* Draft-tree construction                                                   */
/* ------------------------------------------------------------------------ */

/* Builds the draft tree that the verify calls take ([README] "How it works":
 * a best-first tree of up to `budget` nodes over the top-K branches at each
 * position, the rank-0 chain placed first (chain pre-seed); [PR606] options
 * table: --specla-top-k is the expansion width K, --ddtree-tau a cumulative
 * log-probability pruning margin).  The pages do not write the procedure;
 * this library computes, for every sequence b:
 *   1. per draft position d (0 .. D-1, predicting the token at depth d+1):
 *      logp_d = log-softmax of draft_logits[b][d], and the K tokens with the
 *      largest logits (ties to the lower token id), in that order;
 *   2. the root (node 0, token root_token[b], score 0); then the chain: node
 *      e = 1 .. min(D, budget-1) is the rank-0 token of position e-1, child of
 *      node e-1; a node's score is the sum of logp over its root path;
 *   3. best-first: while fewer than `budget` nodes exist, add the candidate
 *      with the highest score, ties to the lower parent index; the
 *      candidates are, for every node at depth < D, its child of the next
 *      rank not yet in the tree (the child of rank r at depth e scores
 *      parent + logp_{e-1}[rank r]); with tau >= 0 a candidate at depth e is
 *      admitted only if its score >= the chain's score at depth e minus tau
 *      (so the tree may stay below `budget`).
 * Nodes are numbered in insertion order (parent[i] < i), as verify expects.
 * Scores are accumulated in fp32 in path order.
 *   draft_logits [B][D][V] f32 (finite), root_token [B] int32
 *   topk_tok [B][D][K] int32, topk_logp [B][D][K] f32: step 1's result
 *                (written; the tree is built from them)
 *   parent, tokens [B][budget] int32 (-1 past n_nodes), n_nodes [B] int32,
 *   score [B][budget] f32 (0 past n_nodes)
 * Supported: 1 <= D <= 64, 1 <= K <= 8, 1 <= budget <= 64, V a multiple of
 * 4 and >= K.  tau: < 0 = no pruning (NaN is rejected). */
typedef struct {
    int32_t B, D, V, K, budget;
    float tau;
    uint32_t flags; /* 0 */
} dflv_ddtree_desc;

dflv_status dflv_ddtree_build(const dflv_ddtree_desc* desc, const float* draft_logits,
                              const int32_t* root_token, int32_t* topk_tok, float* topk_logp,
                              int32_t* parent, int32_t* tokens, int32_t* n_nodes, float* score,
                              int32_t* status_dev, dflv_stream_t stream);

/* ------------------------------------------------------------------------ */
/* Attention layer                                                           */
/* ------------------------------------------------------------------------ */

/* Shape of one attention layer's verify.  Hq must be a multiple of Hkv;
 * query head h reads KV head h / (Hq / Hkv).  cap = slots per (sequence, KV
 * head) in the cache planes.  window W >= 0: a key at position j is visible
 * to a node at position p iff j <= p and (W == 0 or j > p - W).  Node i sits
 * at position P + depth(i).  scale multiplies q.k (usually 1/sqrt(D)).
 * Supported: 1 <= N_max <= 64; q8_0/q4_0 with D in {64, 128, 256}; the
 * asymmetric types and TQ3_0 with D in {128, 256}; f32 with D a multiple of
 * 4, D <= 256. */
typedef struct {
    int32_t B, N_max, Hq, Hkv, D, cap, window;
    dflv_kv_type type;
    float scale;
    uint32_t flags; /* 0 or DFLV_FLAG_EARLY_PREFETCH */
} dflv_attn_desc;

/* One attention layer's cache, structure-of-arrays planes (each plane in its
 * own format for the asymmetric types):
 *   kq, vq : q8_0: int8 [B][Hkv][cap][D]; q4_0: uint8 [B][Hkv][cap][D/2]
 *            (element j < 16 of a 32-block in the low nibble of byte j,
 *            element j+16 in its high nibble); TQ3_0: uint8
 *            [B][Hkv][cap][3D/8] (12 bytes per 32-block); f32: float
 *            [B][Hkv][cap][D]
 *   ks, vs : fp16 [B][Hkv][cap][D/32] block scales (NULL for f32) */
typedef struct {
    void* kq;
    void* vq;
    uint16_t* ks;
    uint16_t* vs;
} dflv_kv_layer;

/* Tree verify of one attention layer.
 *   parent [B][N_max] int32; n_nodes [B] int32
 *   n_past [B] int32 (device): P, the committed tokens of each sequence
 *   q      [B][N_max][Hq][D] bf16; k_new, v_new [B][N_max][Hkv][D] bf16
 *   cache  host pointer to the layer's planes: slots [P, P + n) are
 *          overwritten with the tree's quantised keys/values (quantiser, per
 *          32-block: d = amax / 127 resp. amax / 7 in fp32, stored as fp16
 *          (round to nearest); codes = round-half-away(x * (1/d)) with the
 *          fp32 reciprocal of the fp32 d, clamped to [-127, 127] resp.
 *          [-8, 7] (+8); slots < P are only read)
 *   out    [B][N_max][Hq][D] f32
 *   workspace, ws_bytes: optional device scratch (16-byte aligned).  With
 *          at least dflv_attn_workspace_size(desc) bytes, the partial
 *          results of the key splits are merged through it (global memory);
 *          with less, or NULL, through the thread-block cluster's shared
 *          memory, which is slower.  The results are the same either way.
 *          Its contents on entry do not matter.  Calls on one stream may
 *          share one workspace; calls that can run at the same time need
 *          their own.
 * Every node attends to the cached positions j < P inside its window and to
 * the tree slots of its ancestors-or-self, reading the quantised values, so
 * a chain tree reproduces sequential decode. */
dflv_status dflv_tree_attn_verify(const dflv_attn_desc* desc, const int32_t* parent,
                                  const int32_t* n_nodes, const int32_t* n_past,
                                  const uint16_t* q, const uint16_t* k_new,
                                  const uint16_t* v_new, const dflv_kv_layer* cache, float* out,
                                  int32_t* status_dev, void* workspace, size_t ws_bytes,
                                  dflv_stream_t stream);

/* Attention tree verify that allocates nothing, for callers that cannot
 * allocate device memory (the pages have no counterpart: this is a
 * deployment aid).  Some hosts forbid device allocation on the path that
 * runs a step: a serving runtime that hands each plugin a fixed memory pool,
 * an allocator that must not be entered while a CUDA graph is being
 * captured, or a latency-bound loop that cannot afford the implicit
 * synchronisation of cudaMalloc.  Such callers use this entry point instead
 * of passing a workspace to dflv_tree_attn_verify.
 *   Arguments and results: exactly those of dflv_tree_attn_verify without
 *   workspace / ws_bytes.  Its merge scratch is one array of
 *   DFLV_NOALLOC_SCRATCH_BYTES in the library's own device memory, which every
 *   GPU that loads the library holds until the process exits.
 *   - A descriptor whose merge needs more scratch than that
 *     (dflv_attn_workspace_size(desc) > DFLV_NOALLOC_SCRATCH_BYTES) returns
 *     DFLV_ERR_CAPACITY and launches nothing.
 *   - It calls no cudaMalloc / cudaFree and no allocating library routine.
 *     The first call on a device looks up the scratch's device address for
 *     that device (with it current); make that first call before any stream
 *     capture.
 *   - Every call on a device shares the one scratch array, which keeps the
 *     last call's contents.  Nothing in it needs to start at zero (each
 *     call writes every value it reads), but calls whose kernels can
 *     overlap on the GPU (other streams, or other host threads) race on it:
 *     run them on one stream, one after the other. */
#define DFLV_NOALLOC_SCRATCH_BYTES (16u << 20)
dflv_status dflv_tree_attn_verify_noalloc(const dflv_attn_desc* desc, const int32_t* parent,
                                          const int32_t* n_nodes, const int32_t* n_past,
                                          const uint16_t* q, const uint16_t* k_new,
                                          const uint16_t* v_new, const dflv_kv_layer* cache, float* out,
                                          int32_t* status_dev, dflv_stream_t stream);

/* Bytes of workspace with which dflv_tree_attn_verify merges through global
 * memory for this descriptor (0: the shape never uses one; also 0 for an
 * invalid descriptor).  The launch plan behind it follows the current
 * device, so query it with the device current that will run the calls. */
size_t dflv_attn_workspace_size(const dflv_attn_desc* desc);

/* ------------------------------------------------------------------------ */
/* Greedy acceptance                                                         */
/* ------------------------------------------------------------------------ */

/* best[b][i] = argmax_v logits[b][i][v] (ties: lowest v; a NaN logit counts
 * as -infinity, so a row of NaN or -infinity gives 0).  Then from the
 * root: while a child c of the current node has tokens[b][c] == best of the
 * current node, move to the lowest-index such c.  path[b][0..L) = visited
 * nodes (path[b][0] = 0), path_len[b] = L >= 1 = tokens committed this
 * step, next_token[b] = best of the last visited node.
 *   logits [B][N_max][vocab] f32; tokens, parent [B][N_max] int32
 *   path, best [B][N_max] int32; path_len, next_token [B] int32
 * Everything stays on the device, so accept -> commit needs no host sync. */
dflv_status dflv_accept_greedy(int32_t B, int32_t N_max, int32_t vocab, const float* logits,
                               const int32_t* tokens, const int32_t* parent,
                               const int32_t* n_nodes, int32_t* path, int32_t* path_len,
                               int32_t* next_token, int32_t* best, int32_t* status_dev,
                               dflv_stream_t stream);

/* ------------------------------------------------------------------------ */
/* Commit / rollback                                                         */
/* ------------------------------------------------------------------------ */

/* Commits the accepted path of every sequence into all layers in one launch.
 *   gdn, n_gdn      : GDN shape (may be NULL when n_gdn == 0)
 *   states          : host array of n_gdn device state pointers (in/out)
 *   factors         : host array of n_gdn factor sets written by verify
 *   attn, n_attn    : attention shape (may be NULL when n_attn == 0)
 *   caches          : host array of n_attn cache plane sets (in/out)
 *   path, path_len  : [B][N_max], [B] int32 from dflv_accept_greedy
 *   n_past          : [B] int32, advanced in place by path_len
 * GDN: S <- e^{g_e} S + sum_{m<L} e^{g_e - g_{p_m}} u_{p_m} k_{p_m}^T with
 * p_m = path[m], e = path[L-1]: the state of the path's end node.  KV: slot
 * P + path[m] moves to P + m for every m < L (all moves read before any
 * write).  Slots [P + L, P + N_max) are left unspecified.  Rejected nodes
 * need no work: verify never wrote the committed state or slots < P.
 * The path must be a root-to-node path of the verified tree (as accept
 * produces); N_max must equal the verify calls' N_max.  path_len[b] must lie
 * in [1, N_max] and every path node in [0, N_max): otherwise DFLV_DEV_PATH is
 * raised, sequence b's states and cache slots are left as they were, and its
 * n_past is unspecified. */
dflv_status dflv_commit_rollback(const dflv_gdn_desc* gdn, int32_t n_gdn, float* const* states,
                                 const dflv_gdn_factors* factors, const dflv_attn_desc* attn,
                                 int32_t n_attn, const dflv_kv_layer* caches,
                                 const int32_t* path, const int32_t* path_len, int32_t* n_past,
                                 int32_t* status_dev, dflv_stream_t stream);

/* Most layers one dflv_commit_rollback call takes (per kind). */
#define DFLV_MAX_COMMIT_GDN_LAYERS 128
#define DFLV_MAX_COMMIT_ATTN_LAYERS 64

/* Human-readable name of a status code (static string). */
const char* dflv_status_string(dflv_status s);

#ifdef __cplusplus
}
#endif
#endif /* DFLV_H */
