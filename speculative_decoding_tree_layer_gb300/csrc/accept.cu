// accept.cu -- greedy acceptance of a verified draft tree.
//
// The DDTree verify skeleton stays argmax ("Luce DFlash" README, "Scope and
// limits"), and the acceptance length counts the tokens committed per
// draft/verify step (README, "Results").  Step 1 finds the target argmax of
// every node (ties: lowest vocab index); step 2 walks from the root while a
// child carries the argmax token of the current node (several: lowest node
// index).  Path, length and the next root token stay on the device, so
// commit can follow without a host round trip.
//
// Step 1 is the HBM-bound part (N x vocab fp32 logits): a thread-block
// cluster per node row splits the vocabulary, each CTA streams its share with
// 16-byte loads, and the cluster reduces (value, index) pairs through
// distributed shared memory -- no global scratch.  Step 2 is one warp per
// sequence: lanes test children in parallel and a ballot picks the lowest
// matching index.
#include <climits>

#include "cluster.cuh"
#include "common.cuh"
#include "kernels.h"

namespace dflv {

namespace {

constexpr int kArgmaxThreads = 512;

// (v, i) beats (bv, bi): larger value, or equal value and lower index.  A
// NaN counts as -infinity, so an all-NaN row gives its lowest index.
DFLV_DEVINL void better(float v, int i, float& bv, int& bi) {
    v = (v != v) ? -INFINITY : v;
    if (v > bv || (v == bv && i < bi)) {
        bv = v;
        bi = i;
    }
}

__global__ void __launch_bounds__(kArgmaxThreads) accept_argmax_kernel(AcceptArgs a, int CS) {
    __shared__ float red_v[kArgmaxThreads / 32];
    __shared__ int red_i[kArgmaxThreads / 32];
    const int rank = (int)cluster_ctarank();
    const int i = blockIdx.y, b = blockIdx.z;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    grid_dependency_wait();
    grid_launch_dependents();
    const int n = __ldg(a.n_nodes + b);
    if (n < 1 || n > a.N_max || i >= n) return;  // uniform over the cluster

    const int V = a.vocab;
    const float* row = a.logits + ((size_t)b * a.N_max + i) * V;
    // this CTA's share of the vocabulary, in multiples of 4
    const int per = (((V + CS - 1) / CS) + 3) & ~3;
    const int c0 = min(V, rank * per), c1 = min(V, c0 + per);
    float bv = -INFINITY;
    int bi = INT_MAX;
    if ((V & 3) == 0) {
        const float4* r4 = reinterpret_cast<const float4*>(row);
        const int q0 = c0 >> 2, q1 = c1 >> 2;
        int q = q0 + tid;
        // eight independent 16-byte loads in flight per thread
        for (; q + 7 * kArgmaxThreads < q1; q += 8 * kArgmaxThreads) {
            float4 x[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) x[u] = __ldcs(r4 + q + u * kArgmaxThreads);
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const int base = (q + u * kArgmaxThreads) * 4;
                better(x[u].x, base, bv, bi);
                better(x[u].y, base + 1, bv, bi);
                better(x[u].z, base + 2, bv, bi);
                better(x[u].w, base + 3, bv, bi);
            }
        }
        for (; q < q1; q += kArgmaxThreads) {
            const float4 x = __ldcs(r4 + q);
            const int base = q * 4;
            better(x.x, base, bv, bi);
            better(x.y, base + 1, bv, bi);
            better(x.z, base + 2, bv, bi);
            better(x.w, base + 3, bv, bi);
        }
    } else {
        for (int c = c0 + tid; c < c1; c += kArgmaxThreads) better(__ldcs(row + c), c, bv, bi);
    }
#pragma unroll
    for (int o = 16; o; o >>= 1) {
        const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
        const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
        better(ov, oi, bv, bi);
    }
    if (lane == 0) {
        red_v[warp] = bv;
        red_i[warp] = bi;
    }
    __syncthreads();
    if (tid == 0) {
        for (int w = 1; w < kArgmaxThreads / 32; ++w) better(red_v[w], red_i[w], bv, bi);
        red_v[0] = bv;
        red_i[0] = bi;
    }
    cluster_sync_all();
    if (rank == 0 && tid == 0) {
        for (int q = 1; q < CS; ++q) {
            const float ov = ld_dsmem_f32(map_to_rank(smem_u32(&red_v[0]), q));
            const int oi = ld_dsmem_s32(map_to_rank(smem_u32(&red_i[0]), q));
            better(ov, oi, bv, bi);
        }
        a.best[(size_t)b * a.N_max + i] = bi;
    }
    cluster_sync_all();  // keep this CTA's shared memory alive for rank 0
}

__global__ void accept_walk_kernel(AcceptArgs a) {
    const int b = blockIdx.x, lane = threadIdx.x;
    grid_dependency_wait();
    grid_launch_dependents();
    const int n = __ldg(a.n_nodes + b), N = a.N_max;
    if (n < 1 || n > N) {
        if (lane == 0) {
            a.path_len[b] = 0;
            raise_status(a.status, DFLV_DEV_TOPOLOGY);
        }
        return;
    }
    const int c0 = lane, c1 = lane + 32;
    const int p0 = c0 < n ? __ldg(a.parent + (size_t)b * N + c0) : -2;
    const int p1 = c1 < n ? __ldg(a.parent + (size_t)b * N + c1) : -2;
    bool bad = false;
    if (c0 < n) bad |= (c0 == 0) ? (p0 != -1) : (p0 < 0 || p0 >= c0);
    if (c1 < n) bad |= (p1 < 0 || p1 >= c1);
    if (__any_sync(0xffffffffu, bad)) {
        if (lane == 0) {
            a.path_len[b] = 0;
            raise_status(a.status, DFLV_DEV_TOPOLOGY);
        }
        return;
    }
    const int t0 = c0 < n ? __ldg(a.tokens + (size_t)b * N + c0) : -1;
    const int t1 = c1 < n ? __ldg(a.tokens + (size_t)b * N + c1) : -1;
    const int b0 = c0 < n ? a.best[(size_t)b * N + c0] : -1;
    const int b1 = c1 < n ? a.best[(size_t)b * N + c1] : -1;
    int cur = 0, L = 1;
    if (lane == 0) a.path[(size_t)b * N] = 0;
    for (;;) {
        const int bc = (cur < 32) ? __shfl_sync(0xffffffffu, b0, cur) : __shfl_sync(0xffffffffu, b1, cur - 32);
        const unsigned m0 = __ballot_sync(0xffffffffu, c0 < n && p0 == cur && t0 == bc);
        const unsigned m1 = __ballot_sync(0xffffffffu, c1 < n && p1 == cur && t1 == bc);
        int nxt;
        if (m0) nxt = __ffs(m0) - 1;
        else if (m1) nxt = 32 + __ffs(m1) - 1;
        else break;
        if (lane == 0) a.path[(size_t)b * N + L] = nxt;
        ++L;
        cur = nxt;
    }
    if (lane == 0) {
        a.path_len[b] = L;
        a.next_token[b] = a.best[(size_t)b * N + cur];
    }
}

}  // namespace

cudaError_t launch_accept_greedy(const AcceptArgs& a, cudaStream_t stream) {
    const int sms = sm_count_cached();
    // enough CTAs to cover the SMs a few times, at most 8 per row (portable cluster)
    const long rows = (long)a.B * a.N_max;
    int cs = 1;
    while (cs < 8 && rows * cs < 2L * sms && (long)cs * 2 * kArgmaxThreads * 16 <= a.vocab) cs *= 2;
    cudaError_t e = launch_pdl(accept_argmax_kernel, dim3(cs, a.N_max, a.B), dim3(kArgmaxThreads), 0, stream, cs, a, cs);
    if (e != cudaSuccess) return e;
    return launch_pdl(accept_walk_kernel, dim3(a.B), dim3(32), 0, stream, 1, a);
}

}  // namespace dflv
