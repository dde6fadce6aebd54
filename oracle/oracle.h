/*
 * oracle.h -- plain CPU oracle for the DDTree tree-verify step.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path links, loads or
 * calls this code: only the tests, the package's smoke check and the
 * benchmark's CPU-baseline leg do.  It shares no code, header, table or
 * helper with the CUDA library; the two agree on array layouts because both
 * follow the same written conventions, not because they share a definition.
 *
 * What it computes (sources are the pages "Luce DFlash" server README and
 * lucebox PR #606 "add SpecLA factor-capture speculative decoding"):
 *
 *   - Tree verify of a gated-DeltaNet layer: every draft-tree node's
 *     recurrent state is its parent's state advanced by one gated delta-rule
 *     step ("Luce DFlash" README, "Architecture note": ggml_gated_delta_net
 *     and its _tree variant; "How it works": one target forward verifies the
 *     whole tree via a causal mask derived from parent pointers).  The
 *     recurrence itself is not written on the pages; the oracle uses the
 *     standard gated delta rule
 *         S' = alpha * S * (I - beta k k^T) + beta v k^T,   o = S' q.
 *   - Tree verify of a full-attention layer over a block-quantised KV cache
 *     (README "Asymmetric K/V quantization": q8_0 default, q4_0 at 4.5 bpv),
 *     optionally restricted to a sliding window ("--fa-window N", 0 = full).
 *   - Greedy acceptance ("Scope and limits": the DDTree verify skeleton stays
 *     argmax; "Results": AL = committed tokens per draft/verify step).
 *   - Commit / rollback ("How it works", "Per-step rollback"): after accept
 *     the recurrent state and KV cache equal those of decoding only the
 *     accepted path.
 *   - The tree-aware short convolution before a gated-DeltaNet layer ("How
 *     it works": ggml_ssm_conv_tree reads each node's K-1 window along the
 *     parent chain; the conv window is part of the rolled-back state).  The
 *     pages do not write the op; the oracle uses a depthwise causal conv
 *     (tap K-1 on the current token, no bias, no activation) and commits the
 *     window of the accepted path.
 *
 * Precision: fp64 arithmetic for everything the method computes in floating
 * point; the committed recurrent state is stored as fp32 between steps.  The
 * block quantiser decides integer codes, so it runs in fp32 with correctly
 * rounded operations only (IEEE division and reciprocal, multiplication,
 * round-half-away, fp16 round to nearest even): the same precision the
 * kernels decide them in.
 *
 * Parity status: every function here is pinned by the "not gpu" tests in
 * tests/test_oracle_*.py (closed forms, invariants, brute force and a
 * library cross-check); none is "parity unpinned".
 *
 * Layouts (row-major, outermost first):
 *   parent   [B][N]   int32, parent[0] = -1, 0 <= parent[i] < i
 *   n_nodes  [B]      int32, 1 <= n_nodes[b] <= N
 *   GDN q,k  [B][N][Hk][dk]  bf16 bits; v [B][N][Hv][dv] bf16 bits
 *   beta, log_alpha [B][N][Hv] f32;  state [B][Hv][dv][dk] f32
 *   GDN out  [B][N][Hv][dv] f32
 *   attention q [B][N][Hq][D] bf16; k_new, v_new [B][N][Hkv][D] bf16
 *   cache planes per layer: quants [B][Hkv][cap][D] (int8, q8_0),
 *       [B][Hkv][cap][D/2] (uint8 nibbles, q4_0), [B][Hkv][cap][3D/8] (uint8
 *       three-bit codes, TQ3_0) or [B][Hkv][cap][D] f32;
 *       scales [B][Hkv][cap][D/32] fp16 bits (unused for f32)
 *   attention out [B][N][Hq][D] f32
 *   logits [B][N][V] f32; tokens [B][N] int32
 */
#ifndef DFLV_ORACLE_H
#define DFLV_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

enum { ORC_OK = 0, ORC_ERR_ARG = 1, ORC_ERR_TOPOLOGY = 2, ORC_ERR_CAPACITY = 4 };
/* Cache types; the last two quantise keys and values differently ("Luce
 * DFlash" README, "Asymmetric K/V quantization"): K q8_0 with V q4_0, and
 * K q4_0 with V q8_0. */
enum { ORC_KV_Q8_0 = 0, ORC_KV_Q4_0 = 1, ORC_KV_F32 = 2, ORC_KV_Q8_0_Q4_0 = 3, ORC_KV_Q4_0_Q8_0 = 4,
       ORC_KV_TQ3_0 = 5 };

/* ---- scalar conversions (the oracle's own) ---- */
double orc_bf16_to_double(uint16_t h);
float orc_half_to_float(uint16_t h);
uint16_t orc_float_to_half_rn(float f);

/* ---- tree topology ---- */
/* Validates parent[0..n) and fills depth[n] and the ancestor-or-self sets as
 * bitmasks (n <= 64).  Returns ORC_OK or ORC_ERR_TOPOLOGY. */
int orc_tree_topology(int n, const int32_t* parent, int32_t* depth, uint64_t* anc_self);

/* ---- gated delta rule ---- */
/* One decode step on a dv x dk state held in fp64:
 *   S_out = alpha * S (I - beta k k^T) + beta v k^T,  o = S_out q.
 * S and S_out may not alias. */
void orc_gdn_step(int dv, int dk, const double* S, const double* q, const double* k,
                  const double* v, double beta, double alpha, double* S_out, double* o);

/* Tree verify: state of node i = step(state of parent[i]), root's parent
 * state = the committed state.  If node_states is non-NULL it receives the
 * fp64 state of every node, [B][N][Hv][dv][dk]. */
int orc_tree_gdn_verify(int B, int N, int Hk, int Hv, int dk, int dv,
                        const int32_t* parent, const int32_t* n_nodes,
                        const uint16_t* q, const uint16_t* k, const uint16_t* v,
                        const float* beta, const float* log_alpha, const float* state,
                        float* out, double* node_states);

/* The same outputs computed by replaying every root-to-node path from the
 * committed state on its own (no state shared between nodes). */
int orc_tree_gdn_verify_bruteforce(int B, int N, int Hk, int Hv, int dk, int dv,
                                   const int32_t* parent, const int32_t* n_nodes,
                                   const uint16_t* q, const uint16_t* k, const uint16_t* v,
                                   const float* beta, const float* log_alpha,
                                   const float* state, float* out);

/* Commit of the recurrent state: decode the accepted nodes path[b][0..L) in
 * order from the committed state and store the result (fp32) in place. */
int orc_gdn_commit(int B, int N, int Hk, int Hv, int dk, int dv,
                   const uint16_t* q, const uint16_t* k, const uint16_t* v,
                   const float* beta, const float* log_alpha,
                   const int32_t* path, const int32_t* path_len, float* state);

/* ---- block quantisation (32 values + one fp16 scale) ---- */
void orc_quantize_q8_0(const float* x, int8_t* qs, uint16_t* d16);
void orc_quantize_q4_0(const float* x, uint8_t* nib, uint16_t* d16);
void orc_dequantize_q8_0(const int8_t* qs, uint16_t d16, double* x);
void orc_dequantize_q4_0(const uint8_t* nib, uint16_t d16, double* x);

/* TQ3_0 ("Luce DFlash" README, "Asymmetric K/V quantization": 3.5 bits per
 * value, an FWHT rotation applied to the query and undone on the attention
 * output when the keys are TQ3_0).  The pages give neither the block layout,
 * the codebook nor the rotation size; the readings here: a block of 32
 * values holds one fp16 scale d = amax / 3 and 32 three-bit codes
 * c = clamp(round_half_away(x * (1/d)), -4, 3) + 4 (12 bytes, code j in bits
 * 3j .. 3j+2 of the little-endian 96-bit block), x = d * (c - 4); the
 * rotation is the orthonormal Walsh-Hadamard transform over the whole head
 * dimension (a power of two), applied to keys AND values before they are
 * quantised (the output can only be rotated back if the values were rotated
 * too), to the query, and again to the output (the orthonormal transform is
 * its own inverse). */
void orc_quantize_tq3_0(const float* x, uint8_t* codes, uint16_t* d16);
void orc_dequantize_tq3_0(const uint8_t* codes, uint16_t d16, double* x);
/* The rotation in fp32, in place (it decides the stored codes): butterflies
 * of stride 1, 2, 4, ..., n/2 in that order, each (a, b) -> (a + b, a - b),
 * then one multiplication by the fp32 value of 1/sqrt(n). */
void orc_fwht_f32(int n, float* x);

/* ---- attention tree verify ---- */
/* Writes the quantised tree keys/values into cache slots [P, P+n) and then
 * attends every (node, query head) to the visible keys.  n_past[b] = P.
 * With rows == NULL every output row is computed; otherwise only the n_rows
 * flat rows (b * N + i) * Hq + h listed (for sampled checks at full size). */
int orc_tree_attn_verify(int B, int N, int Hq, int Hkv, int D, int cap, int window,
                         int kv_type, double scale,
                         const int32_t* parent, const int32_t* n_nodes, const int32_t* n_past,
                         const uint16_t* q, const uint16_t* k_new, const uint16_t* v_new,
                         void* kq, void* vq, uint16_t* ks, uint16_t* vs, float* out,
                         const int32_t* rows, int n_rows);

/* ---- greedy acceptance ---- */
int orc_accept_greedy(int B, int N, int V, const float* logits, const int32_t* tokens,
                      const int32_t* parent, const int32_t* n_nodes,
                      int32_t* path, int32_t* path_len, int32_t* next_token, int32_t* best);

/* ---- tree-aware short convolution ---- */
/* Depthwise causal convolution of width K over the tree ("Luce DFlash"
 * README, "How it works": ggml_ssm_conv_tree, each node reads its K-1 window
 * along the DDTree parent chain).  Window position K-1 is node i itself,
 * K-2 its parent, and so on; once the chain has passed the root, the
 * positions read the conv state, the K-1 inputs before the root (state
 * entry K-2 just before the root, entry 0 the oldest):
 *   out[b][i][c] = sum_{j<K} w[c][j] * window_j[c].
 * x [B][N][C] and state [B][K-1][C] are bf16 bits, w [C][K] f32, out
 * [B][N][C] f32 (fp64 sums). */
int orc_tree_conv_verify(int B, int N, int C, int K, const int32_t* parent, const int32_t* n_nodes,
                         const uint16_t* x, const uint16_t* state, const float* w, float* out);

/* Conv state commit: the state becomes the last K-1 entries of the sequence
 * [state ; x of path[b][0..L)], i.e. what decoding the accepted nodes in
 * order would leave behind. */
int orc_conv_commit(int B, int N, int C, int K, const uint16_t* x, const int32_t* path,
                    const int32_t* path_len, uint16_t* state);

/* Threads used by the functions that loop over independent (sequence, head)
 * or output rows (OpenMP when compiled with it): sets n (> 0) and returns
 * the count in force.  Results do not depend on it. */
int orc_set_threads(int n);

/* ---- KV commit: move slot P+path[m] to P+m for m < L (all reads first) ---- */
int orc_kv_commit(int B, int N, int Hkv, int D, int cap, int kv_type,
                  const int32_t* path, const int32_t* path_len, const int32_t* n_past,
                  void* kq, void* vq, uint16_t* ks, uint16_t* vs);

#ifdef __cplusplus
}
#endif
#endif
