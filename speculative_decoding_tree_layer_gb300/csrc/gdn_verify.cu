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
// every row of S_0 is independent: a CTA owns RB rows of one head, streams
// them from HBM once through the bulk-copy (TMA) engine, forms
// S_0[rows] . [K | Q] on the tensor cores (fp32 state split into bf16 hi +
// lo, k and q exact in bf16), then solves the unit lower-triangular system
// for u by substitution over the tree's depth levels (all nodes of a level
// at once, one warp per node, lanes over rows) and mixes the outputs.  It
// writes u, g and a copy of k as the factors commit needs, and never writes
// S_0 (rollback is free).
#include "common.cuh"
#include "kernels.h"
#include "tree.cuh"

namespace dflv {

namespace {

constexpr int kGdnThreads = 256;
constexpr int kGdnWarps = kGdnThreads / 32;

struct GdnSmemLayout {
    int NP, DK, RB, KS;
    size_t off_S, off_V, off_K, off_Q, off_A, off_M, off_R, off_SQ, total;
    __host__ __device__ GdnSmemLayout(int np, int dk, int rb) : NP(np), DK(dk), RB(rb), KS(dk + 16) {
        off_S = 3200;  // header: mbarrier + per-node arrays (3136 B), rounded up to 128
        off_V = off_S + (size_t)RB * DK * 4;     // bf16 v of this CTA's rows, [node][RB]
        off_K = off_V + (size_t)NP * RB * 2;
        off_Q = off_K + (size_t)NP * KS * 2;
        off_A = off_Q + (size_t)NP * KS * 2;
        off_M = off_A + (size_t)NP * NP * 4;
        off_R = off_M + (size_t)NP * NP * 4;
        off_SQ = off_R + (size_t)NP * RB * 4;
        total = off_SQ + (size_t)NP * RB * 4;
    }
};

// sum over the set bits l of m of w[l] * x[l * stride], four terms at a time
// so the shared-memory loads of a group are in flight together
DFLV_DEVINL float masked_dot(uint64_t m, const float* __restrict__ w, const float* __restrict__ x, int stride) {
    float acc = 0.f;
    while (m) {
        int l[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            l[k] = m ? ffs64(m) : -1;
            m &= m - 1;
        }
        float wv[4], xv[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            wv[k] = l[k] >= 0 ? w[l[k]] : 0.f;
            xv[k] = l[k] >= 0 ? x[l[k] * stride] : 0.f;
        }
#pragma unroll
        for (int k = 0; k < 4; ++k) acc = fmaf(wv[k], xv[k], acc);
    }
    return acc;
}

template <int DK, int RB>
__global__ void __launch_bounds__(kGdnThreads)
    gdn_tree_verify_kernel(GdnVerifyArgs a, int NP) {
    extern __shared__ __align__(128) unsigned char smem[];
    const GdnSmemLayout L(NP, DK, RB);
    constexpr int KS = DK + 16;  // bf16 row stride: conflict-free 8-byte fragment loads

    uint64_t* bar = reinterpret_cast<uint64_t*>(smem);
    int32_t* misc_s = reinterpret_cast<int32_t*>(smem + 16);  // [0] = deepest level
    int32_t* par_s = reinterpret_cast<int32_t*>(smem + 64);
    int32_t* depth_s = par_s + kMaxNodes;
    int32_t* order_s = depth_s + kMaxNodes;           // nodes sorted by depth
    int32_t* lvl_s = order_s + kMaxNodes;             // first index of each level in order_s (65)
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

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int gq = lane >> 2, tq = lane & 3;  // MMA fragment row group / thread in quad
    const int b = blockIdx.z, h = blockIdx.y, r0 = blockIdx.x * RB;
    const int N = a.N_max;
    const int hk = h / (a.Hv / a.Hk);

    if (tid == 0) {
        mbar_init(bar, 1);
        fence_mbar_init();
        misc_s[0] = 0;
    }
    __syncthreads();
    grid_dependency_wait();

    // 1. Every input of this CTA is requested at once: its RB rows of S_0
    //    (contiguous) through the bulk-copy engine, and the parent array, the
    //    node scalars, keys, queries and v block with 16- / 4-byte cp.async.
    //    All N_max node rows are fetched (rows past n are never read back
    //    into a result), so nothing waits for n.
    if (tid == 0) {
        const float* src = a.state + (((size_t)b * a.Hv + h) * a.dv + r0) * DK;
        mbar_arrive_expect_tx(bar, RB * DK * 4);
        bulk_g2s(S_s, src, RB * DK * 4, bar);
    }
    constexpr int CH = DK / 8;  // 16-byte chunks per bf16 row
    for (int idx = tid; idx < N * CH; idx += kGdnThreads) {
        const int i = idx / CH, c = idx % CH;
        const size_t off = (((size_t)b * N + i) * a.Hk + hk) * DK + c * 8;
        cp_async16(K_s + i * KS + c * 8, a.k + off);
        cp_async16(Q_s + i * KS + c * 8, a.q + off);
    }
    constexpr int VCH = RB / 8;  // 16-byte chunks of this CTA's v rows
    for (int idx = tid; idx < N * VCH; idx += kGdnThreads) {
        const int i = idx / VCH, c = idx % VCH;
        cp_async16(V_s + i * RB + c * 8, a.v + (((size_t)b * N + i) * a.Hv + h) * a.dv + r0 + c * 8);
    }
    for (int i = tid; i < N; i += kGdnThreads) {
        const size_t sidx = ((size_t)b * N + i) * a.Hv + h;
        cp_async4(beta_s + i, a.beta + sidx);
        cp_async4(la_s + i, a.log_alpha + sidx);
        cp_async4(par_s + i, a.parent + (size_t)b * N + i);
    }
    cp_async_commit();
    // rows [N, NP) of K and Q take part in the tensor-core tiles: zero them
    for (int idx = tid; idx < (NP - N) * CH; idx += kGdnThreads) {
        const int i = N + idx / CH, c = idx % CH;
        *reinterpret_cast<uint4*>(K_s + i * KS + c * 8) = make_uint4(0, 0, 0, 0);
        *reinterpret_cast<uint4*>(Q_s + i * KS + c * 8) = make_uint4(0, 0, 0, 0);
    }
    const int n = __ldg(a.n_nodes + b);
    cp_async_wait<0>();
    __syncthreads();

    // 2. Tree topology (from the staged parent array).
    if (!block_tree_topology_smem(n, N, par_s, depth_s, amask_s, a.status)) {
        if (tid == 0) mbar_wait_bounded(bar, 0, a.status);  // let the copy land before leaving
        return;
    }

    // 3. Nodes ordered by depth (level d = order_s[lvl_s[d] .. lvl_s[d+1])).
    for (int i = tid; i < n; i += kGdnThreads) {
        const int d = depth_s[i];
        int pos = 0;
        for (int j = 0; j < n; ++j) {
            const int dj = depth_s[j];
            pos += (dj < d) || (dj == d && j < i);
        }
        order_s[pos] = i;
        atomicMax(misc_s, d);
    }
    __syncthreads();
    const int maxd = misc_s[0];
    for (int d = tid; d <= maxd + 1; d += kGdnThreads) {
        int c = 0;
        for (int j = 0; j < n; ++j) c += depth_s[j] < d;
        lvl_s[d] = c;
    }
    // cumulative log decay over the ancestors-or-self
    for (int i = tid; i < n; i += kGdnThreads) {
        float g = 0.f;
        for (uint64_t m = amask_s[i]; m; m &= m - 1) g += la_s[ffs64(m)];
        g_s[i] = g;
        G_s[i] = expf(g);
    }

    // 4. [K ; Q] K^T on the tensor cores: KK (rows < NP) and KQ (rows >= NP).
    //    The MMA's k index is permuted consistently on both operands: thread
    //    tq of a quad holds columns 4tq .. 4tq+3 of each 16-wide k step, so
    //    one 8-byte load fills both halves of its fragment registers.
    {
        const int nt_count = NP / 8, tiles = (2 * NP / 16) * nt_count;
        for (int tile = warp; tile < tiles; tile += kGdnWarps) {
            const int mt = tile / nt_count, nt = tile % nt_count;
            const uint16_t* Ap = (mt * 16 < NP) ? K_s + (mt * 16) * KS : Q_s + (mt * 16 - NP) * KS;
            const uint16_t* Bp = K_s + (nt * 8 + gq) * KS;
            float d[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int ks = 0; ks < DK / 16; ++ks) {
                const int col = ks * 16 + tq * 4;
                const uint2 a0 = *reinterpret_cast<const uint2*>(Ap + gq * KS + col);
                const uint2 a1 = *reinterpret_cast<const uint2*>(Ap + (gq + 8) * KS + col);
                const uint2 bb = *reinterpret_cast<const uint2*>(Bp + col);
                const uint32_t af[4] = {a0.x, a1.x, a0.y, a1.y};
                const uint32_t bf[2] = {bb.x, bb.y};
                mma_bf16_16816(d, af, bf);
            }
            const int row = mt * 16 + gq, col = nt * 8 + tq * 2;
            float* dst = (row < NP) ? A_s + row * NP : M_s + (row - NP) * NP;
            dst[col] = d[0];
            dst[col + 1] = d[1];
            dst[8 * NP + col] = d[2];
            dst[8 * NP + col + 1] = d[3];
        }
    }
    __syncthreads();

    // 5. Decays and the ancestor mask:
    //    A_il = beta_i e^{g_i-g_l} k_i.k_l (l strict ancestor), M_il = e^{g_i-g_l} q_i.k_l (l in anc*(i)).
    for (int idx = tid; idx < n * n; idx += kGdnThreads) {
        const int i = idx / n, l = idx % n;
        const bool anc = (amask_s[i] >> l) & 1ull;
        const float dec = anc ? expf(g_s[i] - g_s[l]) : 0.f;
        A_s[i * NP + l] = (anc && l != i) ? beta_s[i] * dec * A_s[i * NP + l] : 0.f;
        M_s[i * NP + l] = anc ? dec * M_s[i * NP + l] : 0.f;
    }

    // 6. S_0[rows] . [K | Q] on the tensor cores, fp32 state as bf16 hi + lo.
    if (!mbar_wait_bounded(bar, 0, a.status)) return;
    {
        constexpr int WM = RB / 16;            // m tiles (16 rows each)
        constexpr int WN = kGdnWarps / WM;     // warps sharing one m tile
        const int mt = warp % WM, wn = warp / WM;
        const int ntiles = 2 * NP / 8;
        constexpr int kMaxJ = (2 * kMaxNodes / 8 + WN - 1) / WN;
        float acc[kMaxJ][4];
#pragma unroll
        for (int j = 0; j < kMaxJ; ++j) acc[j][0] = acc[j][1] = acc[j][2] = acc[j][3] = 0.f;
        const float* S0 = S_s + (mt * 16 + gq) * DK;
        const float* S8 = S0 + 8 * DK;
#pragma unroll 2
        for (int ks = 0; ks < DK / 16; ++ks) {
            const int col = ks * 16 + tq * 4;
            const float4 s0 = *reinterpret_cast<const float4*>(S0 + col);
            const float4 s1 = *reinterpret_cast<const float4*>(S8 + col);
            uint32_t ahi[4], alo[4];
            split_bf16x2(s0.x, s0.y, ahi[0], alo[0]);
            split_bf16x2(s1.x, s1.y, ahi[1], alo[1]);
            split_bf16x2(s0.z, s0.w, ahi[2], alo[2]);
            split_bf16x2(s1.z, s1.w, ahi[3], alo[3]);
#pragma unroll
            for (int j = 0; j < kMaxJ; ++j) {
                const int nt = wn + WN * j;
                if (nt < ntiles) {
                    const uint16_t* Bp = (nt * 8 < NP) ? K_s + (nt * 8 + gq) * KS
                                                       : Q_s + (nt * 8 - NP + gq) * KS;
                    const uint2 bb = *reinterpret_cast<const uint2*>(Bp + col);
                    const uint32_t bf[2] = {bb.x, bb.y};
                    mma_bf16_16816(acc[j], ahi, bf);
                    mma_bf16_16816(acc[j], alo, bf);
                }
            }
        }
        // SK -> R_s[node][row], SQ -> SQ_s[node][row]
#pragma unroll
        for (int j = 0; j < kMaxJ; ++j) {
            const int nt = wn + WN * j;
            if (nt < ntiles) {
                const int c = nt * 8 + tq * 2, row = mt * 16 + gq;
                float* dst = (c < NP) ? R_s + c * RB : SQ_s + (c - NP) * RB;
                dst[row] = acc[j][0];
                dst[RB + row] = acc[j][1];
                dst[row + 8] = acc[j][2];
                dst[RB + row + 8] = acc[j][3];
            }
        }
    }
    __syncthreads();

    // 7. R_j = beta_j (v_j - e^{g_j} S_0 k_j) for this CTA's rows.
    for (int idx = tid; idx < n * RB; idx += kGdnThreads) {
        const int j = idx / RB, r = idx % RB;
        const float vv = bf16_bits_to_float(V_s[j * RB + r]);
        R_s[j * RB + r] = beta_s[j] * (vv - G_s[j] * R_s[j * RB + r]);
    }
    __syncthreads();

    // 8. u_i = R_i - sum_{l in anc(i)} A_il u_l, level by level (a node's
    //    ancestors sit on shallower levels); R_s becomes U in place.
    for (int d = 1; d <= maxd; ++d) {
        const int l0 = lvl_s[d], l1 = lvl_s[d + 1];
        for (int idx = l0 * RB + tid; idx < l1 * RB; idx += kGdnThreads) {
            const int i = order_s[idx / RB], r = idx % RB;
            const uint64_t m = amask_s[i] & ~(1ull << i);
            R_s[i * RB + r] -= masked_dot(m, A_s + i * NP, R_s + r, RB);
        }
        __syncthreads();
    }

    // 9. o_i = e^{g_i} SQ_i + sum_{l in anc*(i)} M_il u_l; u and o to global.
    for (int idx = tid; idx < n * RB; idx += kGdnThreads) {
        const int i = idx / RB, r = idx % RB;
        const float O = G_s[i] * SQ_s[i * RB + r] + masked_dot(amask_s[i], M_s + i * NP, R_s + r, RB);
        const size_t off = (((size_t)b * N + i) * a.Hv + h) * a.dv + r0 + r;
        a.u[off] = R_s[i * RB + r];
        a.out[off] = O;
    }

    // 10. The remaining factors, once per (sequence, head) / (sequence, q/k head).
    if (blockIdx.x == 0) {
        for (int i = tid; i < n; i += kGdnThreads) a.g[((size_t)b * N + i) * a.Hv + h] = g_s[i];
        if (h % (a.Hv / a.Hk) == 0)
            for (int idx = tid; idx < n * CH; idx += kGdnThreads) {
                const int i = idx / CH, c = idx % CH;
                *reinterpret_cast<uint4*>(a.kcopy + (((size_t)b * N + i) * a.Hk + hk) * DK + c * 8) =
                    *reinterpret_cast<const uint4*>(K_s + i * KS + c * 8);
            }
    }
}

template <int DK, int RB>
cudaError_t launch_dk_rb(const GdnVerifyArgs& a, cudaStream_t stream) {
    const int NP = ((a.N_max + 15) / 16) * 16;
    const GdnSmemLayout L(NP, DK, RB);
    auto kern = gdn_tree_verify_kernel<DK, RB>;
    cudaError_t e = ensure_smem(kern, L.total);
    if (e != cudaSuccess) return e;
    dim3 grid(a.dv / RB, a.Hv, a.B);
    kern<<<grid, kGdnThreads, L.total, stream>>>(a, NP);
    return cudaGetLastError();
}

template <int DK>
cudaError_t launch_dk(const GdnVerifyArgs& a, cudaStream_t stream) {
    if (a.dv % 32 == 0) return launch_dk_rb<DK, 32>(a, stream);
    return launch_dk_rb<DK, 16>(a, stream);
}

}  // namespace

size_t gdn_verify_smem_bytes(int N_max, int dk, int dv) {
    const int NP = ((N_max + 15) / 16) * 16;
    return GdnSmemLayout(NP, dk, dv % 32 == 0 ? 32 : 16).total;
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
