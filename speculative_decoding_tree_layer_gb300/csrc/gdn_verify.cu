// gdn_verify.cu -- tree verify of one gated-DeltaNet layer.
//
// What it computes (see include/dflv.h): for every node i of the draft tree
// and every v-head h,
//     S_i = alpha_i S_par(i) (I - beta_i k_i k_i^T) + beta_i v_i k_i^T,   o_i = S_i q_i,
// with the committed state S_0 as the root's parent state.  The pages name
// the tree-mode op ("Luce DFlash" README, "Architecture note":
// ggml_gated_delta_net_tree, which rolls the SSM state back in place) and
// the reason to avoid materialising per-node states (README, "How it works":
// ggml_gated_delta_net_tree_persist writes intermediates directly instead of
// a 9 ms copy; SpecLA PR #606: factor capture).
//
// How: the WY / UT form of the delta rule with the causal mask replaced by
// the tree's ancestor mask.  With u_i = beta_i (v_i - alpha_i S_par(i) k_i)
// and g_i = sum of log alpha over i's ancestors-or-self,
//     S_i = e^{g_i} S_0 + sum_{l in anc*(i)} e^{g_i - g_l} u_l k_l^T,
//     u_i + sum_{l in anc(i)} A_il u_l = R_i,
//         A_il = beta_i e^{g_i - g_l} (k_i . k_l),   R_i = beta_i v_i - beta_i e^{g_i} (S_0 k_i),
//     o_i = e^{g_i} (S_0 q_i) + sum_{l in anc*(i)} M_il u_l,   M_il = e^{g_i - g_l} (k_l . q_i).
// A and M depend on k, q, beta and the decays only -- not on the state -- so
// every row of S_0 is independent: a CTA owns RB rows of one head and
// streams them from HBM once through the bulk-copy (TMA) engine.  Half of
// its warps form K K^T and Q K^T on the tensor cores (lower-triangular tiles
// only) and apply the decays and the ancestor mask, giving dense
// lower-triangular A and M; the other half form S_0[rows] . [K | Q] on the
// tensor cores (fp32 state split into bf16 hi + lo, k and q exact in bf16).
// Then the unit lower-triangular system for u is solved in node order
// (parent[i] < i) by all threads, several per state row, column by column
// with each u broadcast by a warp shuffle, and the outputs are mixed in the
// same pass (one lane per row and a separate output pass for blocks of
// fewer than 64 rows with trees over 32 nodes).  The node count is padded to a compile-time
// NPT (32 or 64) so every loop has a fixed trip count and the tensor-core
// fragments of a step are loaded together.  With early prefetch the state
// rows and the tree are fetched before the kernel waits for its predecessor,
// and, when every CTA of the launch is resident at once, the layer's k, q, v
// rows and node scalars are requested into the L2.
// It writes u, g and a copy of k as the factors commit needs.  A plain
// verify never writes S_0 (rollback is free); with a pending path (deferred
// commit) a CTA first applies the previous step's accepted path to its rows
// and writes those rows back, so the state is the committed one again.
#include "common.cuh"
#include "kernels.h"
#include "tree.cuh"

namespace dflv {

namespace {

constexpr int kGdnThreads = 256;
constexpr int kGdnWarps = kGdnThreads / 32;
constexpr int kHalfWarps = kGdnWarps / 2;

struct GdnSmemLayout {
    int NP, DK, RB, KS;
    size_t off_S, off_V, off_K, off_Q, off_A, off_M, off_R, off_SQ, off_PK, off_PU, off_PC, total;
    __host__ __device__ GdnSmemLayout(int np, int dk, int rb) : NP(np), DK(dk), RB(rb), KS(dk + 16) {
        off_S = 3200;  // header: mbarrier + per-node arrays (3136 B), rounded up to 128
        off_V = off_S + (size_t)RB * DK * 4;     // bf16 v of this CTA's rows, [node][RB]
        off_K = off_V + (size_t)NP * RB * 2;
        off_Q = off_K + (size_t)NP * KS * 2;
        off_A = off_Q + (size_t)NP * KS * 2;     // dense [NP][NP], zero off the strict ancestors
        off_M = off_A + (size_t)NP * NP * 4;     // dense [NP][NP], zero off the ancestors-or-self
        off_R = off_M + (size_t)NP * NP * 4;     // [node][RB]: S_0 k, then u
        off_SQ = off_R + (size_t)NP * RB * 4;    // [node][RB]: S_0 q
        off_PK = off_SQ + (size_t)NP * RB * 4;   // deferred commit: the previous step's k, [node][KS]
        off_PU = off_PK + (size_t)NP * KS * 2;   // its u for this CTA's rows, [node][RB]
        off_PC = off_PU + (size_t)NP * RB * 4;   // its g per node, then e^{g_e - g_{p_m}} per m, then e^{g_e}
        total = off_PC + (size_t)(2 * 64 + 4) * 4;
    }
};

// barrier over `count` threads of the block (whole warps), id != 0
DFLV_DEVINL void named_barrier_sync(int id, int count) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}
// the arriving half of such a barrier: does not wait (its writes before it
// are visible to the threads that pass the matching bar.sync)
DFLV_DEVINL void named_barrier_arrive(int id, int count) {
    asm volatile("bar.arrive %0, %1;" ::"r"(id), "r"(count) : "memory");
}

// Where A_il and M_il sit in shared memory.  Trees of up to 32 nodes, and
// larger ones with 64-row blocks, are solved by every thread of the block,
// TPR = 256 / RB threads per state row, thread q of a row owning nodes q,
// q + TPR, q + 2 TPR, ...: there both matrices are stored by column l, with
// each thread's nodes contiguous, so a thread reads its share of a column
// with vector loads.  The remaining shapes keep row-major [i][l].
template <int NPT, int RB>
DFLV_DEVINL int amat_at(int i, int l) {
    if constexpr (NPT <= 32 || RB == 64) {
        constexpr int TPR = kGdnThreads / RB, NPN = NPT / TPR;
        return l * NPT + (i % TPR) * NPN + i / TPR;
    } else {
        return i * NPT + l;
    }
}

// 4-5. [K ; Q] K^T on the tensor cores by the kHalfWarps warps of the first
//    half, with the decays and the ancestor mask applied to the accumulators:
//      A_il = beta_i e^{g_i-g_l} k_i.k_l for strict ancestors l of i,
//      M_il = e^{g_i-g_l} q_i.k_l for l in anc*(i), zero elsewhere
//    (including every row of a node >= n).  Only the 16 x 8 tiles that reach
//    the diagonal or below are formed (ancestors have smaller indices), and
//    only those are ever read back.  A warp keeps all of its tiles in flight
//    at once.  The MMA's k index is permuted consistently on both operands:
//    thread tq of a quad holds columns 4tq .. 4tq+3 of each 16-wide k step,
//    so one 8-byte load fills both halves of its fragment registers.  The
//    cumulative decays g_s (written by the other half, which arrives at
//    barrier 1 when done) are read only after that barrier, once the
//    products are in registers.
template <int DK, int NPT, int RB>
DFLV_DEVINL void gdn_gram_tiles(const uint16_t* K_s, const uint16_t* Q_s, float* A_s, float* M_s,
                                const float* g_s, const float* beta_s, const uint64_t* amask_s, int n, int warp,
                                int gq, int tq) {
    constexpr int KS = DK + 16;
    constexpr int MT = NPT / 16;                 // 16-row tiles per half
    constexpr int PER = MT * (MT + 1);           // lower tiles per half: 2m + 2 in tile row m
    constexpr int TPW = 2 * PER / kHalfWarps;    // tiles per warp
    static_assert((2 * PER) % kHalfWarps == 0, "tiles must split evenly over the warps");
    const uint16_t* Ap[TPW];
    const uint16_t* Bp[TPW];
    int row0[TPW], col0[TPW];
    bool isM[TPW];
#pragma unroll
    for (int t = 0; t < TPW; ++t) {
        const int tile = warp + kHalfWarps * t;
        const int half = tile / PER;             // 0: K rows (A), 1: Q rows (M)
        int q = tile % PER, m = 0;
        while (q >= 2 * m + 2) {
            q -= 2 * m + 2;
            ++m;
        }
        const int nt = q;
        Ap[t] = (half ? Q_s : K_s) + (m * 16 + gq) * KS;
        Bp[t] = K_s + (nt * 8 + gq) * KS;
        row0[t] = m * 16 + gq;
        col0[t] = nt * 8 + tq * 2;
        isM[t] = half != 0;
    }
    float d[TPW][4];
#pragma unroll
    for (int t = 0; t < TPW; ++t) d[t][0] = d[t][1] = d[t][2] = d[t][3] = 0.f;
#pragma unroll
    for (int ks = 0; ks < DK / 16; ++ks) {
        const int col = ks * 16 + tq * 4;
        uint2 a0[TPW], a1[TPW], bb[TPW];
#pragma unroll
        for (int t = 0; t < TPW; ++t) {
            a0[t] = *reinterpret_cast<const uint2*>(Ap[t] + col);
            a1[t] = *reinterpret_cast<const uint2*>(Ap[t] + 8 * KS + col);
            bb[t] = *reinterpret_cast<const uint2*>(Bp[t] + col);
        }
#pragma unroll
        for (int t = 0; t < TPW; ++t) {
            const uint32_t af[4] = {a0[t].x, a1[t].x, a0[t].y, a1[t].y};
            const uint32_t bf[2] = {bb[t].x, bb[t].y};
            mma_bf16_16816(d[t], af, bf);
        }
    }
    named_barrier_sync(1, kGdnThreads);  // g_s complete (written by the other half)
#pragma unroll
    for (int t = 0; t < TPW; ++t) {
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const int i = row0[t] + (e >> 1) * 8, l = col0[t] + (e & 1);
            float v = 0.f;
            if (i < n && ((amask_s[i] >> l) & 1ull) && (isM[t] || l != i)) {
                const float dec = expf(g_s[i] - g_s[l]);
                v = isM[t] ? dec * d[t][e] : beta_s[i] * dec * d[t][e];
            }
            (isM[t] ? M_s : A_s)[amat_at<NPT, RB>(i, l)] = v;
        }
    }
}

// 6. S_0[rows] . [K | Q] by the kHalfWarps warps wq of the second half: the
//    fp32 state as bf16 hi + lo against exact bf16 k and q.  SK goes to
//    R_s[node][row], SQ to SQ_s[node][row].  A warp owns one 16-row tile and
//    J column tiles; hi and lo accumulate separately while that keeps the
//    register count low, so no two consecutive MMAs depend on each other.
template <int DK, int RB, int NPT>
DFLV_DEVINL void gdn_state_products(const float* S_s, const uint16_t* K_s, const uint16_t* Q_s, float* R_s,
                                    float* SQ_s, int wq, int gq, int tq) {
    constexpr int KS = DK + 16;
    constexpr int WM = RB / 16;              // m tiles (16 rows each)
    constexpr int WN = kHalfWarps / WM;      // warps sharing one m tile
    static_assert(WM * WN == kHalfWarps, "row block must split over the warps");
    constexpr int J = 2 * NPT / 8 / WN;      // column tiles per warp
    constexpr bool SPLIT = J <= 4;           // separate lo accumulators
    const int mt = wq % WM, wn = wq / WM;
    const uint16_t* Bp[J];
#pragma unroll
    for (int j = 0; j < J; ++j) {
        const int nt = wn + WN * j;
        Bp[j] = (nt * 8 < NPT) ? K_s + (nt * 8 + gq) * KS : Q_s + (nt * 8 - NPT + gq) * KS;
    }
    float acc[J][4], acl[SPLIT ? J : 1][4];
#pragma unroll
    for (int j = 0; j < J; ++j) acc[j][0] = acc[j][1] = acc[j][2] = acc[j][3] = 0.f;
#pragma unroll
    for (int j = 0; j < (SPLIT ? J : 1); ++j) acl[j][0] = acl[j][1] = acl[j][2] = acl[j][3] = 0.f;
    const float* S0 = S_s + (mt * 16 + gq) * DK;
    const float* S8 = S0 + 8 * DK;
#pragma unroll 2
    for (int ks = 0; ks < DK / 16; ++ks) {
        const int col = ks * 16 + tq * 4;
        const float4 s0 = *reinterpret_cast<const float4*>(S0 + col);
        const float4 s1 = *reinterpret_cast<const float4*>(S8 + col);
        uint2 bb[J];
#pragma unroll
        for (int j = 0; j < J; ++j) bb[j] = *reinterpret_cast<const uint2*>(Bp[j] + col);
        uint32_t ahi[4], alo[4];
        split_bf16x2(s0.x, s0.y, ahi[0], alo[0]);
        split_bf16x2(s1.x, s1.y, ahi[1], alo[1]);
        split_bf16x2(s0.z, s0.w, ahi[2], alo[2]);
        split_bf16x2(s1.z, s1.w, ahi[3], alo[3]);
#pragma unroll
        for (int j = 0; j < J; ++j) {
            const uint32_t bf[2] = {bb[j].x, bb[j].y};
            mma_bf16_16816(acc[j], ahi, bf);
        }
#pragma unroll
        for (int j = 0; j < J; ++j) {
            const uint32_t bf[2] = {bb[j].x, bb[j].y};
            if constexpr (SPLIT) mma_bf16_16816(acl[j], alo, bf);
            else mma_bf16_16816(acc[j], alo, bf);
        }
    }
#pragma unroll
    for (int j = 0; j < J; ++j) {
        const int nt = wn + WN * j;
        const int c = nt * 8 + tq * 2, row = mt * 16 + gq;
        float* dst = (c < NPT) ? R_s + c * RB : SQ_s + (c - NPT) * RB;
        float v[4] = {acc[j][0], acc[j][1], acc[j][2], acc[j][3]};
        if constexpr (SPLIT) {
#pragma unroll
            for (int e = 0; e < 4; ++e) v[e] += acl[j][e];
        }
        dst[row] = v[0];
        dst[RB + row] = v[1];
        dst[row + 8] = v[2];
        dst[RB + row + 8] = v[3];
    }
}

// Deferred commit, by the 128 threads of the second half (ht = 0..127):
// S <- e^{g_e} S + sum_{m<PL} e^{g_e - g_{p_m}} u_{p_m} k_{p_m}^T on this CTA's
// rows in shared memory, and the updated rows back to the state in HBM.
// PK_s, PU_s and PC_s[0, 64) hold the previous step's k, u and g of every
// node; p = path.
template <int DK, int RB>
DFLV_DEVINL void gdn_apply_pending(const GdnVerifyArgs& a, float* S_s, const uint16_t* PK_s, const float* PU_s,
                                   float* PC_s, const int32_t* path, int PL, int b, int h, int r0, int ht) {
    constexpr int KS = DK + 16;
    float* PW_s = PC_s + kMaxNodes;  // e^{g_e - g_{p_m}} per m, then e^{g_e}
    const float ge = PC_s[path[PL - 1]];  // g of the path's end node
    if (ht < PL) PW_s[ht] = expf(ge - PC_s[path[ht]]);
    if (ht == 0) PW_s[kMaxNodes] = expf(ge);
    named_barrier_sync(2, kGdnThreads / 2);
    const float Ge = PW_s[kMaxNodes];
    float* dst = a.state_out + (((size_t)b * a.Hv + h) * a.dv + r0) * DK;
    // Thread ht owns the float4 at column c = 4 (ht % (DK/4)) of rows
    // r_j = ht / (DK/4) + j * 128 / (DK/4): the same four columns in every
    // row, so each path node's k contributes one 8-byte load per thread, and
    // the rows' values stay in registers across the path.
    constexpr int C4 = DK / 4;                       // float4 per row
    constexpr int TOT = RB * C4;                     // float4 in the row block
    constexpr int J = (TOT + kGdnThreads / 2 - 1) / (kGdnThreads / 2);
    constexpr int RSTEP = (kGdnThreads / 2) / C4;    // rows between a thread's items
    static_assert((kGdnThreads / 2) % C4 == 0, "a thread keeps one column group");
    const int c = (ht % C4) * 4, rr = ht / C4;
    float4 x[J];
#pragma unroll
    for (int j = 0; j < J; ++j) {
        x[j] = make_float4(0.f, 0.f, 0.f, 0.f);
        if (ht + j * (kGdnThreads / 2) < TOT) {
            x[j] = *reinterpret_cast<const float4*>(S_s + (rr + j * RSTEP) * DK + c);
            x[j].x *= Ge;
            x[j].y *= Ge;
            x[j].z *= Ge;
            x[j].w *= Ge;
        }
    }
    for (int m = 0; m < PL; ++m) {
        const int p = path[m];
        const float wm = PW_s[m];
        const uint2 kk = *reinterpret_cast<const uint2*>(PK_s + p * KS + c);
        const float k0 = bf16_bits_to_float((uint16_t)(kk.x & 0xffff)), k1 = bf16_bits_to_float((uint16_t)(kk.x >> 16));
        const float k2 = bf16_bits_to_float((uint16_t)(kk.y & 0xffff)), k3 = bf16_bits_to_float((uint16_t)(kk.y >> 16));
#pragma unroll
        for (int j = 0; j < J; ++j) {
            const int r = min(rr + j * RSTEP, RB - 1);
            const float w = wm * PU_s[p * RB + r];
            x[j].x = fmaf(w, k0, x[j].x);
            x[j].y = fmaf(w, k1, x[j].y);
            x[j].z = fmaf(w, k2, x[j].z);
            x[j].w = fmaf(w, k3, x[j].w);
        }
    }
#pragma unroll
    for (int j = 0; j < J; ++j) {
        if (ht + j * (kGdnThreads / 2) < TOT) {
            const int r = rr + j * RSTEP;
            *reinterpret_cast<float4*>(S_s + r * DK + c) = x[j];
            *reinterpret_cast<float4*>(dst + r * DK + c) = x[j];
        }
    }
    named_barrier_sync(2, kGdnThreads / 2);  // every row is updated before the products read them
}

template <int DK, int RB, int NPT>
__global__ void __launch_bounds__(kGdnThreads, (NPT == 32 && RB <= 32) ? 3 : 2)
    gdn_tree_verify_kernel(GdnVerifyArgs a) {
    extern __shared__ __align__(128) unsigned char smem[];
    const GdnSmemLayout L(NPT, DK, RB);
    constexpr int KS = DK + 16;  // bf16 row stride: conflict-free 8-byte fragment loads

    uint64_t* bar = reinterpret_cast<uint64_t*>(smem);
    int32_t* misc_s = reinterpret_cast<int32_t*>(smem + 16);  // [1]: the state copy timed out
    int32_t* par_s = reinterpret_cast<int32_t*>(smem + 64);
    int32_t* depth_s = par_s + kMaxNodes;
    int32_t* ppath_s = depth_s + kMaxNodes;  // deferred commit: the pending path
    uint64_t* amask_s = reinterpret_cast<uint64_t*>(smem + 64 + 4 * 256 + 512);
    float* beta_s = reinterpret_cast<float*>(smem + 64 + 4 * 256 + 512 + 512);
    float* la_s = beta_s + kMaxNodes;
    float* g_s = la_s + kMaxNodes;
    float* G_s = g_s + kMaxNodes;
    float* S_s = reinterpret_cast<float*>(smem + L.off_S);
    uint16_t* V_s = reinterpret_cast<uint16_t*>(smem + L.off_V);
    uint16_t* K_s = reinterpret_cast<uint16_t*>(smem + L.off_K);
    uint16_t* Q_s = reinterpret_cast<uint16_t*>(smem + L.off_Q);
    float* A_s = reinterpret_cast<float*>(smem + L.off_A);
    float* M_s = reinterpret_cast<float*>(smem + L.off_M);
    float* R_s = reinterpret_cast<float*>(smem + L.off_R);
    float* SQ_s = reinterpret_cast<float*>(smem + L.off_SQ);
    uint16_t* PK_s = reinterpret_cast<uint16_t*>(smem + L.off_PK);
    float* PU_s = reinterpret_cast<float*>(smem + L.off_PU);
    float* PC_s = reinterpret_cast<float*>(smem + L.off_PC);

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int gq = lane >> 2, tq = lane & 3;  // MMA fragment row group / thread in quad
    const int b = blockIdx.z, h = blockIdx.y, r0 = blockIdx.x * RB;
    const int N = a.N_max;
    const int hk = h / (a.Hv / a.Hk);

    // With early prefetch, everything up to the dependency wait reads only
    // the committed state and the tree, which the preceding kernel does not
    // write; the rest waits for it.
    const bool early = (a.flags & DFLV_FLAG_EARLY_PREFETCH) != 0;
    if (!early) grid_dependency_wait();
    if (tid == 0) {
        mbar_init(bar, 1);
        fence_mbar_init();
        misc_s[1] = 0;
    }
    __syncthreads();

    // 1. This CTA's RB rows of S_0 (contiguous) through the bulk-copy engine,
    //    and the parent array; then, once the inputs of this layer may be
    //    read, the keys, queries, v block and node scalars with 16- / 4-byte
    //    cp.async.  All N_max node rows are fetched (rows past n are never
    //    read back into a result), so nothing waits for n.
    if (tid == 0) {
        const float* src = a.state + (((size_t)b * a.Hv + h) * a.dv + r0) * DK;
        mbar_arrive_expect_tx(bar, RB * DK * 4);
        bulk_g2s(S_s, src, RB * DK * 4, bar);
    }
    for (int i = tid; i < N; i += kGdnThreads) cp_async4(par_s + i, a.parent + (size_t)b * N + i);
    const bool pending = a.pend_path != nullptr;
    constexpr int CH = DK / 8;  // 16-byte chunks per bf16 row
    if (pending) {
        // the pending path and the previous step's k, u (this CTA's rows)
        // and g of every node, all in the same round trip: the path picks
        // its rows from them in shared memory
        for (int i = tid; i < N; i += kGdnThreads) {
            cp_async4(ppath_s + i, a.pend_path + (size_t)b * N + i);
            cp_async4(PC_s + i, a.pend_g + ((size_t)b * N + i) * a.Hv + h);
        }
        if (tid == 0) cp_async4(misc_s + 2, a.pend_len + b);
        constexpr int UCH = RB / 4;  // 16-byte chunks of this CTA's u row block
        for (int idx = tid; idx < N * (CH + UCH); idx += kGdnThreads) {
            const int i = idx / (CH + UCH), c = idx % (CH + UCH);
            if (c < CH)
                cp_async16(PK_s + i * KS + c * 8, a.pend_k + (((size_t)b * N + i) * a.Hk + hk) * DK + c * 8);
            else
                cp_async16(PU_s + i * RB + (c - CH) * 4,
                           a.pend_u + (((size_t)b * N + i) * a.Hv + h) * a.dv + r0 + (c - CH) * 4);
        }
    }
    cp_async_commit();
    // The first half (warps 0-3) requests this layer's inputs; the second
    // half (warps 4-7) fetches the pending commit's rows and brings the state
    // rows up to date -- before the dependency wait with early prefetch, as
    // all of that was written by the previous step.
    const bool gram_half = warp < kHalfWarps;
    const int ht = gram_half ? tid : tid - kGdnThreads / 2;  // thread index within the half
    constexpr int kHalf = kGdnThreads / 2;
    // With early prefetch in a launch whose CTAs are all resident at once,
    // the first half also asks for this layer's inputs in the L2 before the
    // dependency wait (in a model the layer before has just written them
    // there); the copies after the wait read them, so whatever the
    // preceding kernel writes in between is what they get.
    if ((a.flags & kFlagPrefetchInputs) && gram_half) {
        constexpr int kPer = 5;  // k row, q row, v block, beta, log_alpha
        for (int idx = ht; idx < N * kPer; idx += kHalf) {
            const int i = idx / kPer, what = idx % kPer;
            const size_t kqo = (((size_t)b * N + i) * a.Hk + hk) * DK;
            const size_t sidx = ((size_t)b * N + i) * a.Hv + h;
            if (what == 0) prefetch_l2_bulk(a.k + kqo, DK * 2);
            else if (what == 1) prefetch_l2_bulk(a.q + kqo, DK * 2);
            else if (what == 2) prefetch_l2_bulk(a.v + sidx * a.dv + r0, RB * 2);
            else prefetch_l2_line((what == 3 ? a.beta : a.log_alpha) + sidx);
        }
    }
    auto issue_layer_inputs = [&]() {
        for (int idx = ht; idx < N * CH; idx += kHalf) {
            const int i = idx / CH, c = idx % CH;
            const size_t off = (((size_t)b * N + i) * a.Hk + hk) * DK + c * 8;
            cp_async16(K_s + i * KS + c * 8, a.k + off);
            cp_async16(Q_s + i * KS + c * 8, a.q + off);
        }
        constexpr int VCH = RB / 8;  // 16-byte chunks of this CTA's v rows
        for (int idx = ht; idx < N * VCH; idx += kHalf) {
            const int i = idx / VCH, c = idx % VCH;
            cp_async16(V_s + i * RB + c * 8, a.v + (((size_t)b * N + i) * a.Hv + h) * a.dv + r0 + c * 8);
        }
        for (int i = ht; i < N; i += kHalf) {
            const size_t sidx = ((size_t)b * N + i) * a.Hv + h;
            cp_async4(beta_s + i, a.beta + sidx);
            cp_async4(la_s + i, a.log_alpha + sidx);
        }
        cp_async_commit();
    };
    if (!early && gram_half) {
        grid_launch_dependents();
        issue_layer_inputs();
    }
    // rows [N, NPT) of K and Q take part in the tensor-core tiles: zero them
    for (int idx = tid; idx < (NPT - N) * CH; idx += kGdnThreads) {
        const int i = N + idx / CH, c = idx % CH;
        *reinterpret_cast<uint4*>(K_s + i * KS + c * 8) = make_uint4(0, 0, 0, 0);
        *reinterpret_cast<uint4*>(Q_s + i * KS + c * 8) = make_uint4(0, 0, 0, 0);
    }
    const int n = __ldg(a.n_nodes + b);
    if (!early && gram_half) cp_async_wait<1>();
    else cp_async_wait<0>();
    __syncthreads();

    // 2. Tree topology (from the staged parent array).
    if (!block_tree_topology_smem(n, N, par_s, depth_s, amask_s, nullptr)) {
        if (early) grid_dependency_wait();
        cp_async_wait<0>();
        if (tid == 0) {
            raise_status(a.status, DFLV_DEV_TOPOLOGY);
            mbar_wait_bounded(bar, 0, a.status);  // let the copy land before leaving
        }
        return;
    }
    // Deferred commit: the pending path (validated by every thread alike).
    int PL = 0;
    if (pending) {
        const int Lp = misc_s[2];
        bool valid = Lp >= 0 && Lp <= N;
        for (int m = 0; valid && m < Lp; ++m) valid = ppath_s[m] >= 0 && ppath_s[m] < N;
        if (!valid) {
            if (tid == 0) raise_status(a.status, DFLV_DEV_PATH);
        } else {
            PL = Lp;
        }
    }
    if (!gram_half) {
        // the previous step's rows landed with the parent array
        if (!mbar_wait_bounded(bar, 0, a.status)) {
            if (lane == 0) atomicOr(misc_s + 1, 1);
        } else if (PL > 0) {
            gdn_apply_pending<DK, RB>(a, S_s, PK_s, PU_s, PC_s, ppath_s, PL, b, h, r0, ht);
        }
        if (early) grid_dependency_wait();  // before any output is written
    } else {
        if (early) {
            grid_dependency_wait();
            grid_launch_dependents();
            issue_layer_inputs();
        }
        cp_async_wait<0>();
    }
    __syncthreads();  // layer inputs and the up-to-date state rows are in place
    if (misc_s[1]) return;  // the state copy never landed (status already raised)

    if (warp < kHalfWarps) {
        gdn_gram_tiles<DK, NPT, RB>(K_s, Q_s, A_s, M_s, g_s, beta_s, amask_s, n, warp, gq, tq);
    } else {
        // 3. cumulative log decay over the ancestors-or-self, by this half
        //    (which has slack: its state products end before the Gram tiles
        //    do): a masked sum over all NPT slots with a fixed trip count
        //    (the loads are the same address across the warp).  The Gram
        //    half's epilogue waits for it at barrier 1.
        const int ht2 = tid - kGdnThreads / 2;
        for (int i = ht2; i < n; i += kGdnThreads / 2) {
            const uint64_t am = amask_s[i];
            float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int l = 0; l < NPT; ++l) acc[l & 3] += ((am >> l) & 1ull) ? la_s[l] : 0.f;
            const float g = (acc[0] + acc[1]) + (acc[2] + acc[3]);
            g_s[i] = g;
            G_s[i] = expf(g);
            if (blockIdx.x == 0) a.g[((size_t)b * N + i) * a.Hv + h] = g;
        }
        named_barrier_arrive(1, kGdnThreads);
        // the factors kept once per (sequence, head) / (sequence, q/k head),
        // written here, off the end of the launch: g above, the keys here
        if (blockIdx.x == 0 && h % (a.Hv / a.Hk) == 0)
            for (int idx = ht2; idx < n * CH; idx += kGdnThreads / 2) {
                const int i = idx / CH, c = idx % CH;
                *reinterpret_cast<uint4*>(a.kcopy + (((size_t)b * N + i) * a.Hk + hk) * DK + c * 8) =
                    *reinterpret_cast<const uint4*>(K_s + i * KS + c * 8);
            }
        // 6. S_0[rows] . [K | Q]
        gdn_state_products<DK, RB, NPT>(S_s, K_s, Q_s, R_s, SQ_s, warp - kHalfWarps, gq, tq);
    }
    __syncthreads();

    // 7-9. Rows are independent: with R_i = beta_i (v_i - e^{g_i} S_0 k_i),
    //      u_i = R_i - sum_{l < i} A_il u_l   (a node's ancestors precede it),
    //      o_i = e^{g_i} SQ_i + sum_{l <= i} M_il u_l.
    //    A and M are zero off the ancestors, so every trip count is fixed.
    if constexpr (NPT <= 32 || RB == 64) {
        // TPR threads per state row, each owning NPN nodes.  Column by
        // column: once u_l is final (in the thread that owns node l) it is
        // broadcast to the row's threads, and each subtracts A_il u_l from
        // its later nodes and adds M_il u_l to their outputs.  The dependence
        // chain per node is one shuffle and one FMA; the rest of a column's
        // work is spread over all 256 threads.
        constexpr int TPR = kGdnThreads / RB;
        constexpr int NPN = NPT / TPR;
        constexpr int VW = NPN >= 4 ? 4 : NPN;  // vector width of a column share
        static_assert(TPR <= 32 && NPN % VW == 0 && (VW == 2 || VW == 4), "row threads within a warp");
        const int r = tid / TPR, q = tid % TPR;
        const int src0 = lane & ~(TPR - 1);
        float x[NPN], o[NPN];  // R_i, then u_i; the output o_i
#pragma unroll
        for (int j = 0; j < NPN; ++j) {
            const int i = q + TPR * j;
            x[j] = 0.f;  // padded nodes keep u = 0
            o[j] = 0.f;
            if (i < n) {
                x[j] = beta_s[i] * (bf16_bits_to_float(V_s[i * RB + r]) - G_s[i] * R_s[i * RB + r]);
                o[j] = G_s[i] * SQ_s[i * RB + r];
            }
        }
        const float* At = A_s + q * NPN;
        const float* Mt = M_s + q * NPN;
#pragma unroll
        for (int l = 0; l < NPT; ++l) {
            if (l >= n) break;  // u_l = 0 from here on
            const int jl = l / TPR;  // a constant once unrolled
            const float ul = __shfl_sync(0xffffffffu, x[jl], src0 | (l % TPR));
#pragma unroll
            for (int g = jl / VW; g < NPN / VW; ++g) {
                float w[VW], m[VW];
                if constexpr (VW == 4) {
                    const float4 a4 = *reinterpret_cast<const float4*>(At + l * NPT + g * 4);
                    const float4 m4 = *reinterpret_cast<const float4*>(Mt + l * NPT + g * 4);
                    w[0] = a4.x, w[1] = a4.y, w[2] = a4.z, w[3] = a4.w;
                    m[0] = m4.x, m[1] = m4.y, m[2] = m4.z, m[3] = m4.w;
                } else {
                    const float2 a2 = *reinterpret_cast<const float2*>(At + l * NPT + g * 2);
                    const float2 m2 = *reinterpret_cast<const float2*>(Mt + l * NPT + g * 2);
                    w[0] = a2.x, w[1] = a2.y;
                    m[0] = m2.x, m[1] = m2.y;
                }
#pragma unroll
                for (int e = 0; e < VW; ++e) {
                    const int j = g * VW + e;
                    if (j >= jl) {  // earlier nodes of this thread are final
                        x[j] = fmaf(-w[e], ul, x[j]);
                        o[j] = fmaf(m[e], ul, o[j]);
                    }
                }
            }
        }
#pragma unroll
        for (int j = 0; j < NPN; ++j) {
            const int i = q + TPR * j;
            if (i < n) {
                const size_t off = (((size_t)b * N + i) * a.Hv + h) * a.dv + r0 + r;
                a.u[off] = x[j];
                a.out[off] = o[j];
            }
        }
    } else {
        // One lane per state row solves all nodes in index order with u in
        // registers; then every thread of the block takes a share of the
        // outputs.  Nodes go in chunks of 8 with no branch inside a chunk,
        // so the loads of a chunk (rows of A, v, S_0 k) are scheduled ahead
        // of the FMA chain.  Nodes n .. chunk end are set to zero and never
        // stored: a valid node i reads u_l for l < 4 ceil(i/4) only, and u_l
        // with l > i is still zero when node i is solved.
        if (tid < RB) {
            const int r = tid;
            float u[NPT];
#pragma unroll
            for (int i = 0; i < NPT; ++i) u[i] = 0.f;
#pragma unroll
            for (int c = 0; c < NPT / 8; ++c) {
                if (8 * c < n) {
#pragma unroll
                    for (int i = 8 * c; i < 8 * c + 8; ++i) {
                        float acc[4] = {beta_s[i] * (bf16_bits_to_float(V_s[i * RB + r]) - G_s[i] * R_s[i * RB + r]),
                                        0.f, 0.f, 0.f};
                        const float4* Ar = reinterpret_cast<const float4*>(A_s + i * NPT);
#pragma unroll
                        for (int l4 = 0; l4 < (i + 3) / 4; ++l4) {
                            const float4 w = Ar[l4];
                            acc[0] = fmaf(-w.x, u[4 * l4], acc[0]);
                            acc[1] = fmaf(-w.y, u[4 * l4 + 1], acc[1]);
                            acc[2] = fmaf(-w.z, u[4 * l4 + 2], acc[2]);
                            acc[3] = fmaf(-w.w, u[4 * l4 + 3], acc[3]);
                        }
                        u[i] = (i < n) ? (acc[0] + acc[1]) + (acc[2] + acc[3]) : 0.f;
                    }
#pragma unroll
                    for (int i = 8 * c; i < 8 * c + 8; ++i)
                        if (i < n) R_s[i * RB + r] = u[i];
                }
            }
        }
        __syncthreads();
        // rows of R_s past n hold S_0 k (finite) and meet zero entries of M
        for (int idx = tid; idx < n * RB; idx += kGdnThreads) {
            const int i = idx / RB, r = idx % RB;
            const float4* Mr = reinterpret_cast<const float4*>(M_s + i * NPT);
            float acc0 = G_s[i] * SQ_s[i * RB + r], acc1 = 0.f;
            for (int l4 = 0; l4 <= i / 4; ++l4) {
                const float4 w = Mr[l4];
                const int l = 4 * l4;
                acc0 = fmaf(w.x, R_s[l * RB + r], acc0);
                acc1 = fmaf(w.y, R_s[(l + 1) * RB + r], acc1);
                acc0 = fmaf(w.z, R_s[(l + 2) * RB + r], acc0);
                acc1 = fmaf(w.w, R_s[(l + 3) * RB + r], acc1);
            }
            const size_t off = (((size_t)b * N + i) * a.Hv + h) * a.dv + r0 + r;
            a.u[off] = R_s[i * RB + r];
            a.out[off] = acc0 + acc1;
        }
    }

}

// CTAs of this kernel the device holds at once at this shared-memory size
// (queried once per instantiation, after its shared-memory limit is raised;
// 0 when the query fails).
template <int DK, int RB, int NPT>
long resident_ctas(size_t smem) {
    static std::atomic<int> cache{0};  // 0 unknown, -1 failed
    int v = cache.load(std::memory_order_relaxed);
    if (v == 0) {
        int nb = 0;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&nb, gdn_tree_verify_kernel<DK, RB, NPT>, kGdnThreads,
                                                          smem) != cudaSuccess ||
            nb < 1) {
            cudaGetLastError();
            nb = -1;
        }
        cache.store(nb, std::memory_order_relaxed);
        v = nb;
    }
    return v > 0 ? (long)v * sm_count_cached() : 0;
}

template <int DK, int RB, int NPT>
cudaError_t launch_dk_rb(const GdnVerifyArgs& a, cudaStream_t stream) {
    const GdnSmemLayout L(NPT, DK, RB);
    auto kern = gdn_tree_verify_kernel<DK, RB, NPT>;
    cudaError_t e = ensure_smem(kern, L.total);
    if (e != cudaSuccess) return e;
    dim3 grid(a.dv / RB, a.Hv, a.B);
    GdnVerifyArgs b = a;
    b.flags &= ~kFlagPrefetchInputs;
    if ((a.flags & DFLV_FLAG_EARLY_PREFETCH) && (long)grid.x * grid.y * grid.z <= resident_ctas<DK, RB, NPT>(L.total))
        b.flags |= kFlagPrefetchInputs;
    return launch_pdl(kern, grid, dim3(kGdnThreads), L.total, stream, 1, b);
}

template <int DK>
cudaError_t launch_dk(const GdnVerifyArgs& a, cudaStream_t stream) {
    const bool small = a.N_max <= 32;
    // 64 state rows per CTA when dv allows it, so that a head takes dv/64
    // CTAs.  Trees of up to 32 nodes: the launch then stays within one CTA
    // per SM at the common shapes (its slowest CTAs share no SM with another
    // CTA of the same launch).  Larger trees: the CTA's shared memory admits
    // one CTA per SM at 32 rows already, so 64 rows halve the waves and the
    // Gram tiles each CTA repeats for its head.
    if (a.dv % 64 == 0)
        return small ? launch_dk_rb<DK, 64, 32>(a, stream) : launch_dk_rb<DK, 64, 64>(a, stream);
    if (a.dv % 32 == 0)
        return small ? launch_dk_rb<DK, 32, 32>(a, stream) : launch_dk_rb<DK, 32, 64>(a, stream);
    return small ? launch_dk_rb<DK, 16, 32>(a, stream) : launch_dk_rb<DK, 16, 64>(a, stream);
}

}  // namespace

size_t gdn_verify_smem_bytes(int N_max, int dk, int dv) {
    const bool small = N_max <= 32;
    return GdnSmemLayout(small ? 32 : 64, dk, dv % 64 == 0 ? 64 : dv % 32 == 0 ? 32 : 16).total;
}

cudaError_t launch_gdn_tree_verify(const GdnVerifyArgs& a, cudaStream_t stream) {
    switch (a.dk) {
        case 16: return launch_dk<16>(a, stream);
        case 32: return launch_dk<32>(a, stream);
        case 64: return launch_dk<64>(a, stream);
        case 128: return launch_dk<128>(a, stream);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace dflv
