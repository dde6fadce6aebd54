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
// cluster per node row splits the vocabulary (up to 16 CTAs, so that a
// 22-node tree still puts two CTAs on every SM), each thread issues all of
// its 16-byte loads of a batch before it compares, and every CTA pushes its
// (value, index) pair into the first CTA's shared memory -- no global
// scratch, no remote loads on the critical path.  Step 2 is one warp per
// sequence: it reads the tree before its launch dependency resolves, marks
// in parallel every node whose token is its parent's argmax, keeps the
// lowest such child per node, and follows those links from the root.
#include <atomic>
#include <climits>

#include "cluster.cuh"
#include "common.cuh"
#include "kernels.h"

namespace dflv {

namespace {

constexpr int kArgmaxThreads = 256;
constexpr int kArgmaxBatch = 12;  // 16-byte loads in flight per thread
constexpr int kMaxArgmaxCluster = 16;

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
    __shared__ float2 part[kMaxArgmaxCluster];  // rank 0: every CTA's (value, index bits)
    const int rank = (int)cluster_ctarank();
    const int i = blockIdx.y, b = blockIdx.z;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    if (CS > 1) cluster_arrive_relaxed();  // paired with the wait before the push
    const int V = a.vocab;
    const float* row = a.logits + ((size_t)b * a.N_max + i) * V;
    // this CTA's share of the vocabulary, in multiples of 4
    const int per = (((V + CS - 1) / CS) + 3) & ~3;
    const int c0 = min(V, rank * per), c1 = min(V, c0 + per);
    // The share is requested into the L2 before the dependency wait (in a
    // model the LM head before has just written the logits there); the loads
    // after the wait read whatever the lines hold by then.
    if (tid == 0 && (V & 3) == 0 && c1 > c0) prefetch_l2_bulk(row + c0, (uint32_t)(c1 - c0) * 4u);
    grid_dependency_wait();
    grid_launch_dependents();
    const int n = __ldg(a.n_nodes + b);
    if (n < 1 || n > a.N_max || i >= n) {  // uniform over the cluster
        if (CS > 1) cluster_wait();
        return;
    }

    float bv = -INFINITY;
    int bi = INT_MAX;
    if ((V & 3) == 0) {
        const float4* r4 = reinterpret_cast<const float4*>(row);
        const int q1 = c1 >> 2;
        for (int q = (c0 >> 2) + tid; q < q1; q += kArgmaxBatch * kArgmaxThreads) {
            float4 x[kArgmaxBatch];
#pragma unroll
            for (int u = 0; u < kArgmaxBatch; ++u)
                if (q + u * kArgmaxThreads < q1) x[u] = __ldcs(r4 + q + u * kArgmaxThreads);
#pragma unroll
            for (int u = 0; u < kArgmaxBatch; ++u) {
                if (q + u * kArgmaxThreads < q1) {
                    const int base = (q + u * kArgmaxThreads) * 4;
                    better(x[u].x, base, bv, bi);
                    better(x[u].y, base + 1, bv, bi);
                    better(x[u].z, base + 2, bv, bi);
                    better(x[u].w, base + 3, bv, bi);
                }
            }
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
    if (warp == 0) {
        bv = lane < kArgmaxThreads / 32 ? red_v[lane] : -INFINITY;
        bi = lane < kArgmaxThreads / 32 ? red_i[lane] : INT_MAX;
#pragma unroll
        for (int o = 4; o; o >>= 1) {
            const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
            const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
            better(ov, oi, bv, bi);
        }
    }
    if (CS == 1) {
        if (tid == 0) a.best[(size_t)b * a.N_max + i] = bi;
        return;
    }
    cluster_wait();  // every CTA of the cluster has started: rank 0's shared memory exists
    if (tid == 0) st_dsmem_f2(map_to_rank(smem_u32(&part[rank]), 0), bv, __int_as_float(bi));
    // release: the push is visible to rank 0 after its acquire; the other
    // ranks' shared memory is never read, so they leave here
    asm volatile("barrier.cluster.arrive.release.aligned;\n" ::: "memory");
    if (rank != 0) return;
    asm volatile("barrier.cluster.wait.acquire.aligned;\n" ::: "memory");
    if (tid == 0) {
        for (int q = 1; q < CS; ++q) better(part[q].x, __float_as_int(part[q].y), bv, bi);
        a.best[(size_t)b * a.N_max + i] = bi;
    }
}

__global__ void __launch_bounds__(32) accept_walk_kernel(AcceptArgs a) {
    __shared__ int child[64];  // lowest-index child whose token is this node's argmax (64: none)
    __shared__ int bst[64];    // every node's argmax
    const int b = blockIdx.x, lane = threadIdx.x, N = a.N_max;
    // The tree and the tokens are step inputs: they were complete before the
    // argmax kernel passed its own dependency wait, so they may be read
    // before this kernel's.
    const int n = __ldg(a.n_nodes + b);
    const bool n_ok = n >= 1 && n <= N;
    const int c0 = lane, c1 = lane + 32;
    const bool in0 = n_ok && c0 < n, in1 = n_ok && c1 < n;
    const int p0 = in0 ? __ldg(a.parent + (size_t)b * N + c0) : -2;
    const int p1 = in1 ? __ldg(a.parent + (size_t)b * N + c1) : -2;
    const int t0 = in0 ? __ldg(a.tokens + (size_t)b * N + c0) : -1;
    const int t1 = in1 ? __ldg(a.tokens + (size_t)b * N + c1) : -1;
    child[c0] = 64;
    child[c1] = 64;
    grid_dependency_wait();
    grid_launch_dependents();
    bool bad = !n_ok;
    if (in0) bad |= (c0 == 0) ? (p0 != -1) : (p0 < 0 || p0 >= c0);
    if (in1) bad |= (p1 < 0 || p1 >= c1);
    if (__any_sync(0xffffffffu, bad)) {
        if (lane == 0) {
            a.path_len[b] = 0;
            raise_status(a.status, DFLV_DEV_TOPOLOGY);
        }
        return;
    }
    const int b0 = in0 ? a.best[(size_t)b * N + c0] : -1;
    const int b1 = in1 ? a.best[(size_t)b * N + c1] : -1;
    // each node's parent's argmax (parents precede their children, so p < n)
    const int q0 = __shfl_sync(0xffffffffu, b0, p0 & 31), r0 = __shfl_sync(0xffffffffu, b1, p0 & 31);
    const int q1 = __shfl_sync(0xffffffffu, b0, p1 & 31), r1 = __shfl_sync(0xffffffffu, b1, p1 & 31);
    bst[c0] = b0;
    bst[c1] = b1;
    __syncwarp();
    if (in0 && c0 > 0 && t0 == (p0 < 32 ? q0 : r0)) atomicMin(&child[p0], c0);
    if (in1 && t1 == (p1 < 32 ? q1 : r1)) atomicMin(&child[p1], c1);
    __syncwarp();
    if (lane == 0) {
        int cur = 0, L = 1;
        a.path[(size_t)b * N] = 0;
        for (int nx = child[0]; nx < 64; nx = child[nx]) {
            a.path[(size_t)b * N + L] = nx;
            ++L;
            cur = nx;
        }
        a.path_len[b] = L;
        a.next_token[b] = bst[cur];
    }
}

// Whether this device can hold a cluster of 16 argmax CTAs (asked once per
// device; the answer also enables the non-portable size for the kernel).
bool cluster16_ok() {
    static std::atomic<int> cache[64];  // 0 unknown, 1 yes, 2 no
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return false;
    int v = cache[dev].load(std::memory_order_relaxed);
    if (v == 0) {
        v = 2;
        if (cudaFuncSetAttribute(accept_argmax_kernel, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) ==
            cudaSuccess) {
            cudaLaunchConfig_t cfg = {};
            cfg.gridDim = dim3(16, 1, 1);
            cfg.blockDim = dim3(kArgmaxThreads, 1, 1);
            cudaLaunchAttribute attr[1];
            attr[0].id = cudaLaunchAttributeClusterDimension;
            attr[0].val.clusterDim.x = 16;
            attr[0].val.clusterDim.y = 1;
            attr[0].val.clusterDim.z = 1;
            cfg.attrs = attr;
            cfg.numAttrs = 1;
            int n_clusters = 0;
            if (cudaOccupancyMaxActiveClusters(&n_clusters, accept_argmax_kernel, &cfg) == cudaSuccess &&
                n_clusters >= 1)
                v = 1;
        }
        cudaGetLastError();
        cache[dev].store(v, std::memory_order_relaxed);
    }
    return v == 1;
}

}  // namespace

cudaError_t launch_accept_greedy(const AcceptArgs& a, cudaStream_t stream) {
    const int sms = sm_count_cached();
    // enough CTAs to put two on every SM, each with at least half a batch
    // of loads per thread; 16 per row uses the non-portable cluster size
    // when this device can schedule it
    const long rows = (long)a.B * a.N_max;
    int cs = 1;
    while (cs < kMaxArgmaxCluster && rows * cs < 2L * sms &&
           (long)cs * 2 * (kArgmaxThreads * 2 * kArgmaxBatch) <= a.vocab)
        cs *= 2;
    if (cs == 16 && !cluster16_ok()) cs = 8;
    cudaError_t e = launch_pdl(accept_argmax_kernel, dim3(cs, a.N_max, a.B), dim3(kArgmaxThreads), 0, stream, cs, a, cs);
    if (e != cudaSuccess) return e;
    return launch_pdl(accept_walk_kernel, dim3(a.B), dim3(32), 0, stream, 1, a);
}

}  // namespace dflv
