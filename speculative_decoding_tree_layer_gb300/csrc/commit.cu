// commit.cu -- commit the accepted path into every layer, in one launch.
//
// After acceptance the recurrent state and the KV cache must equal those of
// decoding only the accepted tokens ("Luce DFlash" README, "How it works",
// per-step rollback; SpecLA PR #606 names the commit routines: compaction of
// the walked path and the pending-factor flush).  Rejected nodes cost nothing
// here because verify never wrote the committed state or the slots below P.
//
//   GDN layer, every (sequence, v-head):  with p_m = path[m], e = path[L-1],
//       S <- e^{g_e} S + sum_{m<L} e^{g_e - g_{p_m}} u_{p_m} k_{p_m}^T,
//   the state of the path's end node in the factor form captured by verify.
//   Each element of S is read and written once (rank-L update in place);
//   the L scaled factor rows sit in shared memory.
//   Attention layer, every (sequence, KV head): slot P + path[m] moves to
//   P + m for m < L.  A destination can be another accepted node's source
//   (path 0, 2, 3: 2 -> 1, 3 -> 2), so the owning CTA reads every source row
//   of a plane into shared memory before it writes any.
// A second tiny kernel then advances n_past by path_len, after every CTA of
// the first has read P.
#include "common.cuh"
#include "kernels.h"

namespace dflv {

namespace {

constexpr int kCommitThreads = 256;

__device__ void commit_gdn_head(const CommitArgs& a, int layer, int b, int h, unsigned char* smem) {
    const int tid = threadIdx.x;
    const CommitGdnLayer ly = a.gdn[layer];
    const int dk = a.dk, dv = a.dv, N = a.N_max;
    float4* S = reinterpret_cast<float4*>(ly.state + ((size_t)b * a.Hv + h) * dv * dk);
    const int E4 = dv * dk / 4;
    constexpr int U = 8;  // float4 per thread in flight
    // The first batch of state loads goes out before the (dependent) factor
    // loads, so their latencies overlap.
    float4 x[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
        const int e4 = u * kCommitThreads + tid;
        if (e4 < E4) x[u] = __ldcs(S + e4);
    }
    // Prologue in two rounds of independent loads: (1) path length and the
    // whole path row, (2) everything indexed by the path.
    __shared__ int32_t path_s[64];
    __shared__ float gp_s[64];
    const int L = __ldg(a.path_len + b);
    const bool L_ok = L >= 1 && L <= N;
    int bad = L_ok ? 0 : 1;
    for (int m = tid; m < N; m += kCommitThreads) {
        const int p = __ldg(a.path + (size_t)b * N + m);
        path_s[m] = p;
        if (L_ok && m < L && (p < 0 || p >= N)) bad = 1;
    }
    if (__syncthreads_or(bad)) {
        if (tid == 0 && layer == 0 && h == 0) raise_status(a.status, DFLV_DEV_PATH);
        return;
    }
    const int hk = h / (a.Hv / a.Hk);
    float* wu_s = reinterpret_cast<float*>(smem);   // [L][dv]  e^{g_e-g_p} u_p
    float* kf_s = wu_s + (size_t)N * dv;            // [L][dk]  k_p
    for (int m = tid; m < L; m += kCommitThreads) gp_s[m] = __ldg(ly.g + ((size_t)b * N + path_s[m]) * a.Hv + h);
    for (int idx = tid; idx < L * dv; idx += kCommitThreads) {
        const int m = idx / dv, r = idx % dv;
        wu_s[idx] = __ldg(ly.u + (((size_t)b * N + path_s[m]) * a.Hv + h) * dv + r);
    }
    for (int idx = tid; idx < L * dk; idx += kCommitThreads) {
        const int m = idx / dk, c = idx % dk;
        kf_s[idx] = bf16_bits_to_float(__ldg(ly.kcopy + (((size_t)b * N + path_s[m]) * a.Hk + hk) * dk + c));
    }
    __syncthreads();
    const float ge = gp_s[L - 1];  // the path's end node
    for (int idx = tid; idx < L * dv; idx += kCommitThreads) wu_s[idx] *= expf(ge - gp_s[idx / dv]);
    __syncthreads();

    const float Ge = expf(ge);
    for (int base = 0; base < E4; base += U * kCommitThreads) {
        if (base > 0) {
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int e4 = base + u * kCommitThreads + tid;
                if (e4 < E4) x[u] = __ldcs(S + e4);
            }
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int e4 = base + u * kCommitThreads + tid;
            if (e4 >= E4) continue;
            const int r = (e4 * 4) / dk, c = (e4 * 4) % dk;
            float4 acc = make_float4(Ge * x[u].x, Ge * x[u].y, Ge * x[u].z, Ge * x[u].w);
            for (int m = 0; m < L; ++m) {
                const float w = wu_s[m * dv + r];
                const float4 kk = *reinterpret_cast<const float4*>(kf_s + m * dk + c);
                acc.x = fmaf(w, kk.x, acc.x);
                acc.y = fmaf(w, kk.y, acc.y);
                acc.z = fmaf(w, kk.z, acc.z);
                acc.w = fmaf(w, kk.w, acc.w);
            }
            __stcs(S + e4, acc);
        }
    }
}

__device__ void commit_kv_head(const CommitArgs& a, int layer, int b, int kvh, unsigned char* smem) {
    const int tid = threadIdx.x;
    const int N = a.N_max;  // <= 64 (the ancestor masks are 64-bit)
    __shared__ int src_s[64];
    // The path length, every path entry and the cache position in one round
    // of loads, then the checks: the path (raised by the GDN heads when
    // there are any) before the capacity.
    const int L = __ldg(a.path_len + b);
    const int P = __ldg(a.n_past + b);
    const bool L_ok = L >= 1 && L <= N;
    bool bad_path = !L_ok, bad_cap = false;
    if (tid < N) {
        const int p = __ldg(a.path + (size_t)b * N + tid);
        if (L_ok && tid < L) {
            if (p < 0 || p >= N) bad_path = true;
            else bad_cap = P + p >= a.cap;
            src_s[tid] = P + p;
        }
    }
    if (__syncthreads_or(bad_path)) {
        if (tid == 0 && layer == 0 && kvh == 0 && a.n_gdn == 0) raise_status(a.status, DFLV_DEV_PATH);
        return;
    }
    if (__syncthreads_or(bad_cap || P < 0 || P + L > a.cap)) {
        if (tid == 0 && kvh == 0) raise_status(a.status, DFLV_DEV_CAPACITY);
        return;
    }
    const CommitAttnLayer ly = a.attn[layer];
    const size_t row0 = ((size_t)b * a.Hkv + kvh) * a.cap;
    // four planes: K codes, V codes, K scales, V scales (no scales for f32);
    // every row is a multiple of 4 bytes (scales: D/32 halves with D >= 64)
    const int planes = a.type == DFLV_KV_F32 ? 2 : 4;
    uint8_t* base[4];
    int w[4], off[4], tot = 0;
#pragma unroll
    for (int pl = 0; pl < 4; ++pl) {
        base[pl] = pl == 0 ? ly.kq : pl == 1 ? ly.vq : reinterpret_cast<uint8_t*>(pl == 2 ? ly.ks : ly.vs);
        w[pl] = pl >= planes ? 0 : (pl < 2 ? kv_code_bytes(a.type, pl, a.D) : a.D / 32 * 2) / 4;
        off[pl] = tot;
        tot += L * w[pl];
    }
    // Every source row of every plane reaches shared memory before any row
    // is written (a destination can be another accepted node's source); the
    // copies of all planes are in flight at once.
    uint32_t* tmp = reinterpret_cast<uint32_t*>(smem);
#pragma unroll
    for (int pl = 0; pl < 4; ++pl)
        for (int idx = tid; idx < L * w[pl]; idx += kCommitThreads) {
            const int m = idx / w[pl], c = idx % w[pl];
            cp_async4(tmp + off[pl] + idx,
                      reinterpret_cast<const uint32_t*>(base[pl] + (row0 + src_s[m]) * (size_t)(4 * w[pl])) + c);
        }
    cp_async_commit();
    cp_async_wait<0>();
    __syncthreads();
#pragma unroll
    for (int pl = 0; pl < 4; ++pl)
        for (int idx = tid; idx < L * w[pl]; idx += kCommitThreads) {
            const int m = idx / w[pl], c = idx % w[pl];
            reinterpret_cast<uint32_t*>(base[pl] + (row0 + P + m) * (size_t)(4 * w[pl]))[c] = tmp[off[pl] + idx];
        }
}

__global__ void __launch_bounds__(kCommitThreads) commit_kernel(const __grid_constant__ CommitArgs a) {
    extern __shared__ __align__(16) unsigned char smem[];
    grid_dependency_wait();
    const int n_gdn_blocks = a.n_gdn * a.B * a.Hv;
    int blk = blockIdx.x;
    if (blk < n_gdn_blocks) {
        const int layer = blk / (a.B * a.Hv), rem = blk % (a.B * a.Hv);
        commit_gdn_head(a, layer, rem / a.Hv, rem % a.Hv, smem);
    } else {
        blk -= n_gdn_blocks;
        const int layer = blk / (a.B * a.Hkv), rem = blk % (a.B * a.Hkv);
        commit_kv_head(a, layer, rem / a.Hkv, rem % a.Hkv, smem);
    }
}

__global__ void commit_advance_kernel(const int32_t* path_len, int32_t* n_past, int B, int N_max) {
    grid_dependency_wait();
    const int b = blockIdx.x * blockDim.x + threadIdx.x;
    if (b >= B) return;
    const int L = path_len[b];
    if (L >= 1 && L <= N_max) n_past[b] += L;
}

}  // namespace

cudaError_t launch_commit_rollback(const CommitArgs& a, cudaStream_t stream) {
    const long blocks = (long)a.n_gdn * a.B * a.Hv + (long)a.n_attn * a.B * a.Hkv;
    if (blocks > 0) {
        size_t smem = 0;
        if (a.n_gdn > 0) smem = (size_t)a.N_max * (a.dv + a.dk) * 4;
        if (a.n_attn > 0) {
            // every plane's rows of the path at once
            const int row_bytes = kv_code_bytes(a.type, 0, a.D) + kv_code_bytes(a.type, 1, a.D) +
                                  (a.type == DFLV_KV_F32 ? 0 : 2 * (a.D / 32) * 2);
            const size_t kv = (size_t)a.N_max * row_bytes;
            if (kv > smem) smem = kv;
        }
        cudaError_t e = ensure_smem(commit_kernel, smem);
        if (e != cudaSuccess) return e;
        // (commit releases no dependent early: the next kernel may read the
        // states it writes)
        e = launch_pdl(commit_kernel, dim3((unsigned)blocks), dim3(kCommitThreads), smem, stream, 1, a);
        if (e != cudaSuccess) return e;
    }
    if (a.n_past != nullptr) {
        return launch_pdl(commit_advance_kernel, dim3((a.B + 255) / 256), dim3(256), 0, stream, 1, a.path_len,
                          a.n_past, a.B, a.N_max);
    }
    return cudaSuccess;
}

}  // namespace dflv
