// tree.cuh -- the draft tree on the device: validation of the parent array,
// node depths and ancestor-or-self bitmasks, computed by one thread block
// into shared memory.
//
// The tree comes as a parent array in topological order with node 0 the
// root (the last committed token) and parent[i] < i; one target pass then
// verifies every node through a causal mask derived from the parent pointers
// ("Luce DFlash" README, "How it works", DDTree tree verify).  With at most
// 64 nodes the mask of node i is one 64-bit word: bit l set iff l is an
// ancestor of i or i itself.
#pragma once

#include "common.cuh"

namespace dflv {

constexpr int kMaxNodes = 64;

// All threads of the block call this.  Reads parent_b[0..n), validates it,
// and fills par_s / depth_s / amask_s for nodes < n.  Returns false for every
// thread (and raises DFLV_DEV_TOPOLOGY once) if n is outside [1, N_max] or a
// parent is out of order; the caller then leaves without writing outputs.
DFLV_DEVINL bool block_tree_topology(const int32_t* __restrict__ parent_b, int n, int N_max,
                                     int32_t* par_s, int32_t* depth_s, uint64_t* amask_s,
                                     int32_t* status_dev) {
    const int tid = threadIdx.x;
    const bool n_ok = (n >= 1 && n <= N_max && n <= kMaxNodes);
    int bad = n_ok ? 0 : 1;
    if (n_ok) {
        for (int i = tid; i < n; i += blockDim.x) {
            int p = __ldg(parent_b + i);
            par_s[i] = p;
            if (i == 0 ? (p != -1) : (p < 0 || p >= i)) bad = 1;
        }
    }
    bad = __syncthreads_or(bad);
    if (bad) {
        if (tid == 0) raise_status(status_dev, DFLV_DEV_TOPOLOGY);
        return false;
    }
    // Each node walks its own ancestor chain (strictly decreasing indices, so
    // at most depth(i) <= i steps).
    for (int i = tid; i < n; i += blockDim.x) {
        uint64_t m = 1ull << i;
        int d = 0;
        for (int c = par_s[i]; c >= 0; c = par_s[c]) {
            m |= 1ull << c;
            ++d;
        }
        depth_s[i] = d;
        amask_s[i] = m;
    }
    __syncthreads();
    return true;
}

// Same as block_tree_topology, with the parent array already in par_s.
DFLV_DEVINL bool block_tree_topology_smem(int n, int N_max, const int32_t* par_s, int32_t* depth_s,
                                          uint64_t* amask_s, int32_t* status_dev) {
    const int tid = threadIdx.x;
    const bool n_ok = (n >= 1 && n <= N_max && n <= kMaxNodes);
    int bad = n_ok ? 0 : 1;
    if (n_ok)
        for (int i = tid; i < n; i += blockDim.x) {
            const int p = par_s[i];
            if (i == 0 ? (p != -1) : (p < 0 || p >= i)) bad = 1;
        }
    bad = __syncthreads_or(bad);
    if (bad) {
        if (tid == 0) raise_status(status_dev, DFLV_DEV_TOPOLOGY);
        return false;
    }
    for (int i = tid; i < n; i += blockDim.x) {
        uint64_t m = 1ull << i;
        int d = 0;
        for (int c = par_s[i]; c >= 0; c = par_s[c]) {
            m |= 1ull << c;
            ++d;
        }
        depth_s[i] = d;
        amask_s[i] = m;
    }
    __syncthreads();
    return true;
}

}  // namespace dflv
