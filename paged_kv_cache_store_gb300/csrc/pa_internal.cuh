// pa_internal.cuh -- shared device helpers and host plumbing of libpa.
//
// Device side: inline-PTX wrappers for mbarriers, TMA (cp.async.bulk.tensor
// and plain cp.async.bulk), bf16 unpacking, and the device error record.
// Every wait on an mbarrier is bounded in time: after kWaitLimitNs the wait
// gives up, the kernel records PA_DEV_TIMEOUT and unwinds, so a bug cannot
// hang the GPU.
#pragma once

#include <cuda.h>
#include <utility>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/pa.h"

namespace pa {

// ---------------------------------------------------------------------------
// Device error record: {code, where}.  The first error wins.
// ---------------------------------------------------------------------------
struct DevError {
    int code;
    int pad;
    long long where;
};

__device__ __forceinline__ void record_error(DevError *e, int code, long long where) {
    if (e == nullptr) return;
    if (atomicCAS(&e->code, 0, code) == 0) {
        atomicExch(reinterpret_cast<unsigned long long *>(&e->where),
                   static_cast<unsigned long long>(where));
    }
}

// Bounded waits give up after this long (the copies they wait for take
// microseconds).
constexpr unsigned long long kWaitLimitNs = 1000ull * 1000ull * 1000ull;  // 1 s

__device__ __forceinline__ unsigned long long globaltimer_ns() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ uint32_t smem_addr(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ---------------------------------------------------------------------------
// mbarrier
// ---------------------------------------------------------------------------
__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count)
                 : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)),
                 "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// Waits until the phase with the given parity has completed.  Returns false
// if that did not happen within kWaitLimitNs.
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity) {
    const uint32_t a = smem_addr(bar);
    if (mbar_try_wait(a, parity)) return true;
    const unsigned long long t0 = globaltimer_ns();
    while (true) {
#pragma unroll 1
        for (int i = 0; i < 32; ++i)
            if (mbar_try_wait(a, parity)) return true;
        if (globaltimer_ns() - t0 > kWaitLimitNs) return false;
    }
}

// ---------------------------------------------------------------------------
// TMA / bulk copies (global -> shared, completion counted on an mbarrier)
// ---------------------------------------------------------------------------
__device__ __forceinline__ void tma_load_3d(void *dst, const CUtensorMap *map, int c0, int c1, int c2,
                                            uint64_t *bar, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%2, %3, %4}], [%5], %6;" ::"r"(smem_addr(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(smem_addr(bar)),
        "l"(policy)
        : "memory");
}

__device__ __forceinline__ void tma_load_4d(void *dst, const CUtensorMap *map, int c0, int c1, int c2, int c3,
                                            uint64_t *bar, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%2, %3, %4, %5}], [%6], %7;" ::"r"(smem_addr(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(smem_addr(bar)),
        "l"(policy)
        : "memory");
}

__device__ __forceinline__ void bulk_load(void *dst, const void *src, uint32_t bytes, uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_addr(dst)),
        "l"(src), "r"(bytes), "r"(smem_addr(bar))
        : "memory");
}

__device__ __forceinline__ void prefetch_tensormap(const CUtensorMap *map) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

__device__ __forceinline__ uint64_t policy_evict_first() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}

__device__ __forceinline__ uint64_t policy_evict_last() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
    return p;
}

// ---------------------------------------------------------------------------
// Named barriers (a subset of the CTA's warps)
// ---------------------------------------------------------------------------
// Programmatic dependent launch: wait until the grids this one depends on
// have completed and their memory is visible, then let the grids that
// depend on this one be scheduled (they wait on this grid the same way).
__device__ __forceinline__ void pdl_wait_then_release() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

__device__ __forceinline__ void named_bar_sync(int id, int nthreads) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// ---------------------------------------------------------------------------
// bf16 helpers: a 32-bit word holds two bf16 (low element first).
// Widening bf16 -> f32 is a 16-bit shift of the bit pattern.
// ---------------------------------------------------------------------------
__device__ __forceinline__ float bf16lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

__device__ __forceinline__ float fast_exp2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ uint4 ld_shared_v4(uint32_t addr) {
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "r"(addr));
    return v;
}

__device__ __forceinline__ uint2 ld_shared_v2(uint32_t addr) {
    uint2 v;
    asm volatile("ld.shared.v2.u32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(addr));
    return v;
}

}  // namespace pa

// ---------------------------------------------------------------------------
// Host plumbing (defined in pa_abi.cu)
// ---------------------------------------------------------------------------
namespace pa {

// Sets the thread-local message and returns status.
pa_status fail(pa_status status, const char *fmt, ...);
// Maps a CUDA error to PA_ERR_CUDA with a message naming `what`.
pa_status cuda_fail(cudaError_t err, const char *what);
// Checks cudaGetLastError after a launch.
pa_status check_launch(const char *kernel);

// Device address of the error record on the current device (nullptr on failure).
DevError *device_error_ptr();
// Current device's SM count (cached per device).
int sm_count();
// Whether checked mode is on.
bool checked_mode();

// Encodes a 4-D bf16 tensor map over a KV pool [num_slots][num_kv_heads][128]
// viewed as [kv head][half][slot][64] (the strides need not grow with the
// dimension), with box {64, box_rows, 2, 1} and 128-byte swizzle: a box of
// box_rows rows of one kv head lands as [2 halves][box_rows][128 B], so 8
// consecutive rows at one 16-byte column fall in 8 different banks.
pa_status encode_kv_tensor_map_halves(CUtensorMap *map, const void *base, int64_t num_slots,
                                      int32_t num_kv_heads, int32_t box_rows);
// The same view for any [rows][heads][128] bf16 tensor with a row stride
// (bytes, a multiple of 16): box {64, box_rows, box_halves, 1}.  With
// box_halves == 1 a copy fetches one 64-dim half (coordinate 2 picks it).
pa_status encode_halves_map(CUtensorMap *map, const void *base, int64_t num_rows, int64_t row_stride_bytes,
                            int32_t num_heads, int32_t box_rows, int32_t box_halves);
// General 3-D bf16 tensor map: dims {dim0, dim1, dim2} (dim0 contiguous),
// byte strides of dims 1 and 2, box {box0, 1, box2}, optional 128-byte swizzle.
pa_status encode_tensor_map_3d(CUtensorMap *map, const void *base, int64_t dim0, int64_t dim1, int64_t dim2,
                               int64_t stride1_bytes, int64_t stride2_bytes, int32_t box0, int32_t box2,
                               bool swizzle128);

inline bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Launches kernel<<<grid, block, smem, stream>>>(args...) as a programmatic
// dependent launch: the grid may be scheduled while the previous work on the
// stream drains, so the kernel must execute griddepcontrol.wait before it
// touches global memory.
template <typename... KArgs, typename... Args>
pa_status launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                     const char *name, Args &&...args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
    if (e != cudaSuccess) return cuda_fail(e, name);
    return check_launch(name);
}

}  // namespace pa
