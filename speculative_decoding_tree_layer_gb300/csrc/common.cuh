// common.cuh -- small device helpers shared by the libdflv kernels:
// bf16/fp16 packing, warp-level tensor-core MMA, the bulk-copy (TMA) engine
// with mbarrier completion and bounded waits, programmatic dependent launch,
// and the device status word.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/dflv.h"

#define DFLV_DEVINL __device__ __forceinline__

namespace dflv {

// ---------------------------------------------------------------- status
DFLV_DEVINL void raise_status(int32_t* status_dev, int bits) {
    if (status_dev) atomicOr(status_dev, bits);
}

// ---------------------------------------------------------------- packing
DFLV_DEVINL float bf16_bits_to_float(uint16_t b) { return __uint_as_float(((uint32_t)b) << 16); }

// Two floats -> packed bf16x2 (round to nearest even); lo in the low half.
DFLV_DEVINL uint32_t pack_bf16x2(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
}

DFLV_DEVINL uint32_t pack_f16x2(float lo, float hi) {
    __half2 v = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
}

// bf16 x -> (hi, lo) with hi = bf16(x), lo = bf16(x - hi): x ~= hi + lo to
// about 16 significant bits.
DFLV_DEVINL void split_bf16x2(float x0, float x1, uint32_t& hi, uint32_t& lo) {
    __nv_bfloat162 h = __floats2bfloat162_rn(x0, x1);
    float2 hf = __bfloat1622float2(h);
    __nv_bfloat162 l = __floats2bfloat162_rn(x0 - hf.x, x1 - hf.y);
    hi = *reinterpret_cast<uint32_t*>(&h);
    lo = *reinterpret_cast<uint32_t*>(&l);
}

// ---------------------------------------------------------------- MMA
// D(16x8, f32) += A(16x16, bf16, row) * B(16x8, bf16, col).
DFLV_DEVINL void mma_bf16_16816(float (&d)[4], const uint32_t (&a)[4], const uint32_t (&b)[2]) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
        "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};\n"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]));
}

// D(16x8, f32) += A(16x16, f16, row) * B(16x8, f16, col).
DFLV_DEVINL void mma_f16_16816(float (&d)[4], const uint32_t (&a)[4], const uint32_t (&b)[2]) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 "
        "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};\n"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]));
}

DFLV_DEVINL void ldmatrix_x4(uint32_t (&r)[4], uint32_t smem_addr) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(smem_addr));
}

DFLV_DEVINL void ldmatrix_x4_trans(uint32_t (&r)[4], uint32_t smem_addr) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];\n"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(smem_addr));
}

DFLV_DEVINL uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ---------------------------------------------------------------- mbarrier + bulk copy
DFLV_DEVINL void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;\n" ::"r"(smem_u32(bar)), "r"(count));
}

DFLV_DEVINL void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
}

DFLV_DEVINL void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");
}

DFLV_DEVINL void mbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];\n" ::"r"(smem_u32(bar)) : "memory");
}

DFLV_DEVINL void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;\n" ::"r"(smem_u32(bar)),
                 "r"(bytes)
                 : "memory");
}

// One bulk (TMA engine) copy global -> shared, completion counted on bar.
// dst, src 16-byte aligned; bytes a multiple of 16.
DFLV_DEVINL void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];\n" ::"r"(
            smem_u32(dst)),
        "l"(src), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}

// Requests [src, src + bytes) into the L2 (TMA engine; src 16-byte aligned,
// bytes a multiple of 16) and the L2 line holding p.  Neither moves data into
// the SM nor orders anything: a later load still reads whatever the line
// holds when it is made, including writes that reach it after the request.
DFLV_DEVINL void prefetch_l2_bulk(const void* src, uint32_t bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;\n" ::"l"(src), "r"(bytes) : "memory");
}
DFLV_DEVINL void prefetch_l2_line(const void* p) {
    asm volatile("prefetch.global.L2 [%0];\n" ::"l"(p) : "memory");
}

// One bulk (TMA engine) copy shared -> global; src, dst 16-byte aligned,
// bytes a multiple of 16.  bulk_s2g_wait() then waits until every such copy
// of this thread has written its data and orders those writes before this
// thread's later generic accesses (and so before a later release).
DFLV_DEVINL void bulk_s2g(void* dst, const void* src, uint32_t bytes) {
    asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;\n" ::"l"(dst), "r"(smem_u32(src)),
                 "r"(bytes)
                 : "memory");
}
DFLV_DEVINL void bulk_s2g_wait() {
    asm volatile("cp.async.bulk.commit_group;\n" ::: "memory");
    asm volatile("cp.async.bulk.wait_group 0;\n" ::: "memory");
    asm volatile("fence.proxy.async.global;\n" ::: "memory");
}

DFLV_DEVINL bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
        " selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Bounded wait on a phase of bar.  Returns false (and raises
// DFLV_DEV_TIMEOUT) if the phase did not complete within the limit; the
// caller then waits once more (bounded) for its copy and leaves.
constexpr uint32_t kWaitLimit = 1u << 22;

DFLV_DEVINL bool mbar_wait_bounded(uint64_t* bar, uint32_t parity, int32_t* status_dev) {
    for (uint32_t it = 0; it < kWaitLimit; ++it)
        if (mbar_try_wait(bar, parity)) return true;
    raise_status(status_dev, DFLV_DEV_TIMEOUT);
    for (uint32_t it = 0; it < kWaitLimit; ++it)
        if (mbar_try_wait(bar, parity)) break;
    return false;
}

// ---------------------------------------------------------------- cp.async (16 B)
DFLV_DEVINL void cp_async16(void* dst, const void* src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(smem_u32(dst)), "l"(src) : "memory");
}
DFLV_DEVINL void cp_async4(void* dst, const void* src) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;\n" ::"r"(smem_u32(dst)), "l"(src) : "memory");
}
DFLV_DEVINL void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }
template <int N>
DFLV_DEVINL void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;\n" ::"n"(N) : "memory");
}

// ---------------------------------------------------------------- PDL
// Waits until the grids this one depends on (programmatic dependent launch)
// have completed and their memory is visible.  A no-op without PDL.
DFLV_DEVINL void grid_dependency_wait() { asm volatile("griddepcontrol.wait;\n" ::: "memory"); }
// Lets the next kernel on the stream (if launched with PDL) be scheduled
// now.  Every kernel of this library calls it only after its own
// grid_dependency_wait, so at most one predecessor of a kernel can still be
// running while that kernel executes the part before its own wait.
DFLV_DEVINL void grid_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory"); }

// ---------------------------------------------------------------- misc
DFLV_DEVINL int popc64(uint64_t x) { return __popcll(x); }
DFLV_DEVINL int ffs64(uint64_t x) { return __ffsll((long long)x) - 1; }

}  // namespace dflv

// ---------------------------------------------------------------- host-side launch helpers
#include <atomic>
#include <mutex>
#include <utility>

namespace dflv {

// SM count of the current device, queried once per device.
inline int sm_count_cached() {
    static std::atomic<int> cache[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 152;
    int v = cache[dev].load(std::memory_order_relaxed);
    if (v > 0) return v;
    if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || v <= 0) v = 152;
    cache[dev].store(v, std::memory_order_relaxed);
    return v;
}

// Raises a kernel's dynamic shared-memory limit only when a launch needs
// more than was already granted to that kernel on this device, so
// steady-state launches (and stream capture) make no attribute calls.
inline cudaError_t ensure_smem_ptr(const void* kern, size_t bytes) {
    struct Grant {
        const void* kern;
        int dev;
        size_t bytes;
    };
    static std::mutex mu;
    static Grant grants[256];
    static int n_grants = 0;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) dev = 0;
    std::lock_guard<std::mutex> lock(mu);
    Grant* g = nullptr;
    for (int i = 0; i < n_grants; ++i)
        if (grants[i].kern == kern && grants[i].dev == dev) g = &grants[i];
    if (g && bytes <= g->bytes) return cudaSuccess;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
    if (e != cudaSuccess) return e;
    if (g) g->bytes = bytes;
    else if (n_grants < 256) grants[n_grants++] = Grant{kern, dev, bytes};
    return cudaSuccess;
}

template <typename Kernel>
inline cudaError_t ensure_smem(Kernel kern, size_t bytes) {
    return ensure_smem_ptr(reinterpret_cast<const void*>(kern), bytes);
}

// Launches kern<<<grid, block, smem, stream>>>(args...) with programmatic
// dependent launch allowed (the kernel may be scheduled while the preceding
// kernel on the stream finishes; it calls grid_dependency_wait before it
// touches anything that kernel may write) and, if cluster_x > 1, as
// clusters of cluster_x CTAs along x.
template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                              int cluster_x, Args&&... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    int na = 0;
    attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[na].val.programmaticStreamSerializationAllowed = 1;
    ++na;
    if (cluster_x > 1) {
        attr[na].id = cudaLaunchAttributeClusterDimension;
        attr[na].val.clusterDim.x = cluster_x;
        attr[na].val.clusterDim.y = 1;
        attr[na].val.clusterDim.z = 1;
        ++na;
    }
    cfg.attrs = attr;
    cfg.numAttrs = na;
    return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}

}  // namespace dflv
