// conv_tree.cu -- the short causal convolution in front of a gated-DeltaNet
// layer, evaluated on the draft tree, and the commit of its window.
//
// On a tree the convolution window of node i is i itself and its K-1 nearest
// ancestors along the parent chain ("Luce DFlash" README, "How it works":
// ggml_ssm_conv_tree); once the chain has passed the root the window runs
// on into the conv state, the K-1 committed inputs before the root:
//     out[i][c] = sum_{j<K} w[c][j] * win_j(i)[c],  win_{K-1}(i) = x_i,
//     win_{K-1-d}(i) = x of the d-th ancestor, or state[K-1+depth(i)-d].
// The work is a few multiply-adds per byte, so the kernel is a memory
// stream: every input byte is read once from HBM (x and state rows into
// shared memory, taps into registers) and every output written once with
// coalesced 8/16-byte accesses.  A CTA owns 128 channels of one sequence;
// its 8 warps split the nodes (warp q takes nodes q, q+8, ...), so a
// thread's serial work is a few nodes rather than the whole tree.  The
// window table (which shared-memory row feeds which tap of which node) is
// built once per CTA from the parent array and read as a warp-wide
// broadcast.
//
// The commit leaves the state that decoding only the accepted path would
// leave: the last K-1 entries of [state ; x_{p_0} .. x_{p_{L-1}}].  One
// launch covers every layer; each thread reads its channels' new window
// before it writes any of it.
#include "common.cuh"
#include "kernels.h"
#include "tree.cuh"

namespace dflv {

namespace {

constexpr int kConvLanes = 32;                       // channel lanes of a CTA
constexpr int kConvCh = 4;                           // channels per lane: one 8-byte bf16x4 access
constexpr int kConvGroups = 8;                       // node groups: lane l of group q takes nodes q, q+8, ...
constexpr int kConvThreads = kConvLanes * kConvGroups;
constexpr int kConvBlockCh = kConvLanes * kConvCh;   // channels per CTA
constexpr int kCommitThreads = 64;
constexpr int kCommitBlockCh = kCommitThreads * kConvCh;

DFLV_DEVINL void cp_async8(void* dst, const void* src) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 8;\n" ::"r"(smem_u32(dst)), "l"(src) : "memory");
}

DFLV_DEVINL void bf16x4_to_float(uint2 v, float (&f)[4]) {
    f[0] = __uint_as_float(v.x << 16);
    f[1] = __uint_as_float(v.x & 0xffff0000u);
    f[2] = __uint_as_float(v.y << 16);
    f[3] = __uint_as_float(v.y & 0xffff0000u);
}

// grid (ceil(C / 128), B), 256 threads = 32 channel lanes x 8 node groups.
// Dynamic shared memory: the x rows of the CTA's channels for nodes
// [0, N_max), then the K-1 state rows; a row is one uint2 per lane.  Every
// thread copies the rows of its own nodes (and group s < K-1 state row s);
// after one barrier any thread reads any row, since a node's window reaches
// into other groups' nodes.
template <int K>
__global__ void __launch_bounds__(kConvThreads) conv_tree_verify_kernel(const ConvVerifyArgs a) {
    static_assert(K - 1 <= kConvGroups, "one node group per state row");
    __shared__ int32_t par_s[kMaxNodes];
    __shared__ int32_t depth_s[kMaxNodes];
    __shared__ uint64_t amask_s[kMaxNodes];
    __shared__ int32_t win_s[kMaxNodes][K];  // win_s[i][d]: row feeding ancestor distance d
    extern __shared__ uint2 rows_s[];
    const int tid = threadIdx.x, lane = tid % kConvLanes, grp = tid / kConvLanes;
    const int b = blockIdx.y, N = a.N_max, C = a.C;
    const int c0 = blockIdx.x * kConvBlockCh + lane * kConvCh;
    const bool active = c0 < C;
    const bool early = (a.flags & DFLV_FLAG_EARLY_PREFETCH) != 0;
    if (!early) grid_dependency_wait();

    // Step-invariant inputs: the taps (4 channels x K contiguous floats), the
    // conv state rows and the tree.
    float w[K][kConvCh];
    if (active) {
        const float4* wp = reinterpret_cast<const float4*>(a.w + (size_t)c0 * K);
        float t[kConvCh * K];
#pragma unroll
        for (int q = 0; q < K; ++q) {
            const float4 v = __ldg(wp + q);
            t[4 * q] = v.x;
            t[4 * q + 1] = v.y;
            t[4 * q + 2] = v.z;
            t[4 * q + 3] = v.w;
        }
#pragma unroll
        for (int j = 0; j < K; ++j)
#pragma unroll
            for (int cc = 0; cc < kConvCh; ++cc) w[j][cc] = t[cc * K + j];
        if (grp < K - 1)
            cp_async8(rows_s + (N + grp) * kConvLanes + lane, a.state + ((size_t)b * (K - 1) + grp) * C + c0);
    }
    const int n = __ldg(a.n_nodes + b);
    if (!block_tree_topology(a.parent + (size_t)b * N, n, N, par_s, depth_s, amask_s, a.status)) {
        cp_async_commit();
        cp_async_wait<0>();
        return;
    }
    for (int i = tid; i < n; i += kConvThreads) {
        int node = i, past = 0;
#pragma unroll
        for (int d = 0; d < K; ++d) {
            if (node >= 0) {
                win_s[i][d] = node;
                node = par_s[node];
            } else {
                win_s[i][d] = N + (K - 2 - past);  // the (past+1)-th input before the root
                ++past;
            }
        }
    }
    if (early) grid_dependency_wait();
    grid_launch_dependents();

    // The nodes' inputs, all in flight at once.
    if (active)
        for (int i = grp; i < n; i += kConvGroups)
            cp_async8(rows_s + i * kConvLanes + lane, a.x + ((size_t)b * N + i) * C + c0);
    cp_async_commit();
    cp_async_wait<0>();
    __syncthreads();  // rows_s and win_s
    if (!active) return;
#pragma unroll 2
    for (int i = grp; i < n; i += kConvGroups) {
        float acc[kConvCh] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int j = 0; j < K; ++j) {
            float f[kConvCh];
            bf16x4_to_float(rows_s[win_s[i][K - 1 - j] * kConvLanes + lane], f);
#pragma unroll
            for (int cc = 0; cc < kConvCh; ++cc) acc[cc] = fmaf(w[j][cc], f[cc], acc[cc]);
        }
        __stcs(reinterpret_cast<float4*>(a.out + ((size_t)b * N + i) * C + c0),
               make_float4(acc[0], acc[1], acc[2], acc[3]));
    }
}

// grid (ceil(C / 256), B, n_layers), 64 threads.
template <int K>
__global__ void __launch_bounds__(kCommitThreads) conv_commit_kernel(const ConvCommitArgs a) {
    grid_dependency_wait();
    const int tid = threadIdx.x, b = blockIdx.y, layer = blockIdx.z, N = a.N_max, C = a.C;
    const int c0 = blockIdx.x * kCommitBlockCh + tid * kConvCh;
    const int L = __ldg(a.path_len + b);
    bool bad = L < 0 || L > N;
    if (!bad)
        for (int m = 0; m < L; ++m) {
            const int p = __ldg(a.path + (size_t)b * N + m);
            bad |= p < 0 || p >= N;
        }
    if (bad) {
        if (tid == 0 && blockIdx.x == 0 && layer == 0) raise_status(a.status, DFLV_DEV_PATH);
        return;
    }
    if (L == 0 || c0 >= C) return;
    uint2* st = reinterpret_cast<uint2*>(a.state[layer] + (size_t)b * (K - 1) * C + c0);
    const uint16_t* x = a.x[layer];
    // new entry s = entry L + s of [state ; x of the path]
    uint2 nv[K - 1];
#pragma unroll
    for (int s = 0; s < K - 1; ++s) {
        const int src = L + s;
        if (src < K - 1) {
            nv[s] = st[(size_t)src * (C / kConvCh)];
        } else {
            const int p = __ldg(a.path + (size_t)b * N + (src - (K - 1)));
            nv[s] = __ldg(reinterpret_cast<const uint2*>(x + ((size_t)b * N + p) * C + c0));
        }
    }
#pragma unroll
    for (int s = 0; s < K - 1; ++s) st[(size_t)s * (C / kConvCh)] = nv[s];
}

template <int K>
cudaError_t launch_verify_k(const ConvVerifyArgs& a, cudaStream_t stream) {
    const dim3 grid((a.C + kConvBlockCh - 1) / kConvBlockCh, a.B);
    const size_t smem = (size_t)(a.N_max + K - 1) * kConvLanes * sizeof(uint2);
    return launch_pdl(conv_tree_verify_kernel<K>, grid, dim3(kConvThreads), smem, stream, 1, a);
}

template <int K>
cudaError_t launch_commit_k(const ConvCommitArgs& a, cudaStream_t stream) {
    const dim3 grid((a.C + kCommitBlockCh - 1) / kCommitBlockCh, a.B, a.n_layers);
    return launch_pdl(conv_commit_kernel<K>, grid, dim3(kCommitThreads), 0, stream, 1, a);
}

}  // namespace

cudaError_t launch_conv_tree_verify(const ConvVerifyArgs& a, cudaStream_t stream) {
    switch (a.K) {
        case 2: return launch_verify_k<2>(a, stream);
        case 3: return launch_verify_k<3>(a, stream);
        case 4: return launch_verify_k<4>(a, stream);
        case 5: return launch_verify_k<5>(a, stream);
        case 6: return launch_verify_k<6>(a, stream);
        case 7: return launch_verify_k<7>(a, stream);
        case 8: return launch_verify_k<8>(a, stream);
    }
    return cudaErrorInvalidValue;
}

cudaError_t launch_conv_commit(const ConvCommitArgs& a, cudaStream_t stream) {
    switch (a.K) {
        case 2: return launch_commit_k<2>(a, stream);
        case 3: return launch_commit_k<3>(a, stream);
        case 4: return launch_commit_k<4>(a, stream);
        case 5: return launch_commit_k<5>(a, stream);
        case 6: return launch_commit_k<6>(a, stream);
        case 7: return launch_commit_k<7>(a, stream);
        case 8: return launch_commit_k<8>(a, stream);
    }
    return cudaErrorInvalidValue;
}

}  // namespace dflv
