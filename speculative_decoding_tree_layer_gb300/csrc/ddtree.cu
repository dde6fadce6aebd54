// ddtree.cu -- construction of the draft tree on the device.
//
// The draft proposes a distribution over the vocabulary for each of the D
// positions after the last committed token; the tree spans the top-K tokens
// of each position, best-first, up to a node budget, after the rank-0 chain
// has been placed ("Luce DFlash" README, "How it works": DDTree tree
// verify, chain pre-seed; SpecLA PR, options table: --specla-top-k is the
// expansion width, --ddtree-tau a cumulative log-probability pruning
// margin).  Readings (include/dflv.h states them in full): log-probabilities
// are the log-softmax of the logits; a node's score is the sum of the
// log-probabilities on its root path; the children of a depth-d node are the
// top-K tokens of position d+1; pruning compares a candidate with the
// chain's score at the same depth.
//
// Step 1 is the HBM-bound part (D x vocab fp32 logits per sequence): a
// thread-block cluster per position splits the vocabulary; each thread keeps
// a running (max, sum of exponentials), updated once per chunk of 32 values,
// and a sorted top-K list in registers while it streams its share with
// 16-byte loads; lists merge warp-wide by K
// rounds of a shuffle argmax, then across the block in shared memory and
// across the cluster through distributed shared memory.  Step 2 builds the
// tree with one warp per sequence: because a node's children enter in rank
// order (the top-K log-probabilities are sorted), every node offers one
// candidate at a time, so a best-first step is one warp-wide argmax over
// the nodes.
#include <climits>

#include "cluster.cuh"
#include "common.cuh"
#include "kernels.h"

namespace dflv {

namespace {

constexpr int kTopkThreads = 512;
constexpr int kTopkWarps = kTopkThreads / 32;
constexpr float kLog2e = 1.4426950408889634f;

// 2^x by the hardware's approximate base-2 exponential (PTX ex2.approx; a
// few ulp, far inside what a log-sum-exp over the vocabulary needs).
DFLV_DEVINL float ex2(float x) {
    float y;
    asm("ex2.approx.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// (v, i) beats (bv, bi): larger value, or equal value and lower index.
DFLV_DEVINL bool beats(float v, int i, float bv, int bi) { return v > bv || (v == bv && i < bi); }

// Running log-sum-exp state: m = max, s = sum of 2^((x - m) log2 e).
DFLV_DEVINL void lse_merge(float& m, float& s, float m2, float s2) {
    if (m2 == -INFINITY) return;
    if (m == -INFINITY) {
        m = m2;
        s = s2;
        return;
    }
    const float mn = fmaxf(m, m2);
    s = s * ex2((m - mn) * kLog2e) + s2 * ex2((m2 - mn) * kLog2e);
    m = mn;
}

// Insert (x, c) into a list sorted by `beats`; c is larger than every index
// already in the list (each thread scans its indices in increasing order),
// so it goes after equal values.
template <int K>
DFLV_DEVINL void topk_insert(float (&v)[K], int (&ix)[K], float x, int c) {
    if (!(x > v[K - 1])) return;
    v[K - 1] = x;
    ix[K - 1] = c;
#pragma unroll
    for (int j = K - 1; j > 0; --j) {
        if (v[j] > v[j - 1]) {
            const float tv = v[j];
            v[j] = v[j - 1];
            v[j - 1] = tv;
            const int ti = ix[j];
            ix[j] = ix[j - 1];
            ix[j - 1] = ti;
        }
    }
}

// K rounds of a warp argmax over the lanes' list heads: every lane ends with
// the warp's top K in (rv, ri).  The lists are consumed.
template <int K>
DFLV_DEVINL void warp_merge_topk(float (&v)[K], int (&ix)[K], float (&rv)[K], int (&ri)[K]) {
#pragma unroll
    for (int r = 0; r < K; ++r) {
        float bv = v[0];
        int bi = ix[0];
#pragma unroll
        for (int o = 16; o; o >>= 1) {
            const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
            const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
            if (beats(ov, oi, bv, bi)) {
                bv = ov;
                bi = oi;
            }
        }
        rv[r] = bv;
        ri[r] = bi;
        if (ix[0] == bi && bi != INT_MAX) {  // this lane's head won: pop it
#pragma unroll
            for (int j = 0; j + 1 < K; ++j) {
                v[j] = v[j + 1];
                ix[j] = ix[j + 1];
            }
            v[K - 1] = -INFINITY;
            ix[K - 1] = INT_MAX;
        }
    }
}

DFLV_DEVINL void warp_merge_lse(float& m, float& s) {
#pragma unroll
    for (int o = 16; o; o >>= 1) {
        const float om = __shfl_xor_sync(0xffffffffu, m, o);
        const float os = __shfl_xor_sync(0xffffffffu, s, o);
        lse_merge(m, s, om, os);
    }
}

// grid (CS, D, B), clusters of CS along x, 512 threads.
template <int K>
__global__ void __launch_bounds__(kTopkThreads) draft_topk_kernel(const DdtreeArgs a, int CS) {
    __shared__ float wv_s[kTopkWarps][K];
    __shared__ int wi_s[kTopkWarps][K];
    __shared__ float wm_s[kTopkWarps], ws_s[kTopkWarps];
    __shared__ float cv_s[K];
    __shared__ int ci_s[K];
    __shared__ float cm_s, cs_s;
    const int rank = (int)cluster_ctarank();
    const int d = blockIdx.y, b = blockIdx.z;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    grid_dependency_wait();
    grid_launch_dependents();

    const int V = a.V;
    const float4* r4 = reinterpret_cast<const float4*>(a.logits + ((size_t)b * a.D + d) * V);
    // this CTA's share of the vocabulary, in float4 units
    const int Q = V >> 2, per = (Q + CS - 1) / CS;
    const int q0 = min(Q, rank * per), q1 = min(Q, q0 + per);
    float v[K];
    int ix[K];
#pragma unroll
    for (int j = 0; j < K; ++j) {
        v[j] = -INFINITY;
        ix[j] = INT_MAX;
    }
    float m = -INFINITY, s = 0.f;
    // Chunks of 8 float4 per thread, all loads in flight at once (past the
    // share's end they read as -inf).  Per chunk: its max updates the running
    // max once, then every value adds 2^((x - m) log2 e) and is offered to
    // the top-K list (indices increase within and across chunks).
    for (int q = q0 + tid; q < q1; q += 8 * kTopkThreads) {
        float4 x[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            const int qq = q + u * kTopkThreads;
            x[u] = qq < q1 ? __ldcs(r4 + qq) : make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
        }
        float cm = -INFINITY;
#pragma unroll
        for (int u = 0; u < 8; ++u) cm = fmaxf(cm, fmaxf(fmaxf(x[u].x, x[u].y), fmaxf(x[u].z, x[u].w)));
        if (cm > m) {  // the chunk's first value is always in range, so cm is finite
            s *= ex2((m - cm) * kLog2e);
            m = cm;
        }
        const float mb = m * kLog2e;
        float cs[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            cs[0] += ex2(fmaf(x[u].x, kLog2e, -mb));
            cs[1] += ex2(fmaf(x[u].y, kLog2e, -mb));
            cs[2] += ex2(fmaf(x[u].z, kLog2e, -mb));
            cs[3] += ex2(fmaf(x[u].w, kLog2e, -mb));
        }
        s += (cs[0] + cs[1]) + (cs[2] + cs[3]);
        // the top-K list only looks at a chunk whose maximum could enter it
        if (cm > v[K - 1]) {
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const int c = (q + u * kTopkThreads) * 4;
                topk_insert<K>(v, ix, x[u].x, c);
                topk_insert<K>(v, ix, x[u].y, c + 1);
                topk_insert<K>(v, ix, x[u].z, c + 2);
                topk_insert<K>(v, ix, x[u].w, c + 3);
            }
        }
    }

    // warp, then block
    float rv[K];
    int ri[K];
    warp_merge_topk<K>(v, ix, rv, ri);
    warp_merge_lse(m, s);
    if (lane == 0) {
#pragma unroll
        for (int j = 0; j < K; ++j) {
            wv_s[warp][j] = rv[j];
            wi_s[warp][j] = ri[j];
        }
        wm_s[warp] = m;
        ws_s[warp] = s;
    }
    __syncthreads();
    if (warp == 0) {
#pragma unroll
        for (int j = 0; j < K; ++j) {
            v[j] = lane < kTopkWarps ? wv_s[lane][j] : -INFINITY;
            ix[j] = lane < kTopkWarps ? wi_s[lane][j] : INT_MAX;
        }
        m = lane < kTopkWarps ? wm_s[lane] : -INFINITY;
        s = lane < kTopkWarps ? ws_s[lane] : 0.f;
        warp_merge_topk<K>(v, ix, rv, ri);
        warp_merge_lse(m, s);
        if (lane == 0) {
#pragma unroll
            for (int j = 0; j < K; ++j) {
                cv_s[j] = rv[j];
                ci_s[j] = ri[j];
            }
            cm_s = m;
            cs_s = s;
        }
    }
    // across the cluster: rank 0 gathers every CTA's list through DSMEM
    cluster_sync_all();
    if (rank == 0 && warp == 0) {
#pragma unroll
        for (int j = 0; j < K; ++j) {
            v[j] = -INFINITY;
            ix[j] = INT_MAX;
        }
        m = -INFINITY;
        s = 0.f;
        if (lane < CS) {
#pragma unroll
            for (int j = 0; j < K; ++j) {
                v[j] = ld_dsmem_f32(map_to_rank(smem_u32(&cv_s[j]), lane));
                ix[j] = ld_dsmem_s32(map_to_rank(smem_u32(&ci_s[j]), lane));
            }
            m = ld_dsmem_f32(map_to_rank(smem_u32(&cm_s), lane));
            s = ld_dsmem_f32(map_to_rank(smem_u32(&cs_s), lane));
        }
        warp_merge_topk<K>(v, ix, rv, ri);
        warp_merge_lse(m, s);
        const float lse = m + logf(s);
        if (lane < K) {
            float val = rv[0];
            int id = ri[0];
#pragma unroll
            for (int j = 1; j < K; ++j)
                if (lane == j) {
                    val = rv[j];
                    id = ri[j];
                }
            const size_t o = ((size_t)b * a.D + d) * K + lane;
            a.topk_tok[o] = id;
            a.topk_logp[o] = val - lse;
        }
    }
    cluster_sync_all();  // peers keep their shared memory until rank 0 has read it
}

// One warp per sequence.
template <int K>
__global__ void __launch_bounds__(32) ddtree_build_kernel(const DdtreeArgs a) {
    __shared__ int tok_s[kMaxTreeDepth * K];
    __shared__ float lp_s[kMaxTreeDepth * K];
    __shared__ float chain_s[kMaxTreeDepth + 1];
    __shared__ int par_s[64], dep_s[64], nr_s[64], tk_s[64];
    __shared__ float sc_s[64];
    const int b = blockIdx.x, lane = threadIdx.x;
    grid_dependency_wait();
    grid_launch_dependents();
    const int D = a.D, N = a.budget;
    for (int e = lane; e < D * K; e += 32) {
        tok_s[e] = a.topk_tok[(size_t)b * D * K + e];
        lp_s[e] = a.topk_logp[(size_t)b * D * K + e];
    }
    __syncwarp();
    if (lane == 0) {  // the chain's score per depth, in path order
        float c = 0.f;
        chain_s[0] = 0.f;
        for (int e = 1; e <= D; ++e) {
            c += lp_s[(e - 1) * K];
            chain_s[e] = c;
        }
    }
    __syncwarp();
    // the root and the chain seed: nodes 0 .. n_chain
    const int n_chain = min(D, N - 1);
    for (int i = lane; i <= n_chain; i += 32) {
        par_s[i] = i - 1;
        dep_s[i] = i;
        sc_s[i] = chain_s[i];
        tk_s[i] = i == 0 ? __ldg(a.root_token + b) : tok_s[(i - 1) * K];
        nr_s[i] = (i == n_chain && n_chain < D) ? 0 : 1;  // a chain node's rank-0 child is the next one
    }
    __syncwarp();
    const bool prune = a.tau >= 0.f;
    int n = n_chain + 1;
    while (n < N) {
        // every node offers its next rank; one warp argmax picks the best
        float bv = -INFINITY;
        int bp = INT_MAX;
        for (int p = lane; p < n; p += 32) {
            const int r = nr_s[p], dd = dep_s[p] + 1;
            if (dd > D || r >= K) continue;
            const float sv = sc_s[p] + lp_s[(dd - 1) * K + r];
            if (prune && sv < chain_s[dd] - a.tau) continue;
            if (beats(sv, p, bv, bp)) {
                bv = sv;
                bp = p;
            }
        }
#pragma unroll
        for (int o = 16; o; o >>= 1) {
            const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
            const int op = __shfl_xor_sync(0xffffffffu, bp, o);
            if (beats(ov, op, bv, bp)) {
                bv = ov;
                bp = op;
            }
        }
        if (bp == INT_MAX) break;  // nothing admissible is left
        if (lane == 0) {
            const int r = nr_s[bp], dd = dep_s[bp] + 1;
            par_s[n] = bp;
            dep_s[n] = dd;
            sc_s[n] = bv;
            tk_s[n] = tok_s[(dd - 1) * K + r];
            nr_s[n] = 0;
            nr_s[bp] = r + 1;
        }
        __syncwarp();
        ++n;
    }
    for (int i = lane; i < N; i += 32) {
        const size_t o = (size_t)b * N + i;
        a.parent[o] = i < n ? par_s[i] : -1;
        a.tokens[o] = i < n ? tk_s[i] : -1;
        a.score[o] = i < n ? sc_s[i] : 0.f;
    }
    if (lane == 0) a.n_nodes[b] = n;
}

template <int K>
cudaError_t launch_k(const DdtreeArgs& a, cudaStream_t stream) {
    const int sms = sm_count_cached();
    const long rows = (long)a.B * a.D;
    int cs = 1;
    while (cs < 8 && rows * cs < 2L * sms && (long)cs * 2 * kTopkThreads * 16 <= a.V) cs *= 2;
    cudaError_t e = launch_pdl(draft_topk_kernel<K>, dim3(cs, a.D, a.B), dim3(kTopkThreads), 0, stream, cs, a, cs);
    if (e != cudaSuccess) return e;
    return launch_pdl(ddtree_build_kernel<K>, dim3(a.B), dim3(32), 0, stream, 1, a);
}

}  // namespace

cudaError_t launch_ddtree_build(const DdtreeArgs& a, cudaStream_t stream) {
    switch (a.K) {
        case 1: return launch_k<1>(a, stream);
        case 2: return launch_k<2>(a, stream);
        case 3: return launch_k<3>(a, stream);
        case 4: return launch_k<4>(a, stream);
        case 5: return launch_k<5>(a, stream);
        case 6: return launch_k<6>(a, stream);
        case 7: return launch_k<7>(a, stream);
        case 8: return launch_k<8>(a, stream);
    }
    return cudaErrorInvalidValue;
}

}  // namespace dflv
