// Internal helpers shared by the libdspark kernels (sm_103a only).
#pragma once

#include <cuda_runtime.h>
#include <cstdint>

#include "dspark.h"

namespace dspark {

// ---- host-side error reporting (common.cu) -------------------------------------------
dspark_status fail(dspark_status s, const char *fmt, ...);
dspark_status cuda_fail(cudaError_t e, const char *what);
void clear_error();
// SM count of the current device (cached per device).
int current_sm_count(int *sm_count);

// Checked probe enqueue behind dspark_conf_probe / dspark_conf_probe_split (probe.cu).  With
// set_cond != 0 the kernel also sets the graph conditional `cond` to probe 0's gate.
dspark_status probe_enqueue(const void *w_q8_0, const float *xa, int Ka, long long lda, const float *xb, int Kb,
                            long long ldb, float bias, float threshold, int n_probes, float *logit_out,
                            int32_t *gate_out, cudaStream_t stream, cudaGraphConditionalHandle cond, int set_cond);

inline bool aligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

// Device status word bits (stored in the workspace header).
constexpr unsigned kStatusIndex = 1u;
constexpr unsigned kStatusTimeout = 2u;

// Default limit for every device-side wait: far above any legitimate wait (a whole
// draft takes well under a millisecond) and short enough to never look like a hang.
constexpr unsigned long long kDefaultTimeoutNs = 2000000000ull;  // 2 s

// ---- device helpers -----------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_addr(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ unsigned long long global_timer_ns() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_addr(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Wait for the phase of `bar` with the given parity to complete; false after
// `timeout_ns` without completion.
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity, unsigned long long timeout_ns) {
    if (mbar_try_wait(bar, parity)) return true;
    const unsigned long long t0 = global_timer_ns();
    while (!mbar_try_wait(bar, parity)) {
        if (global_timer_ns() - t0 > timeout_ns) return false;
    }
    return true;
}

__device__ __forceinline__ uint64_t l2_policy_evict_first() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}

__device__ __forceinline__ uint64_t l2_policy_evict_last() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
    return p;
}

// Programmatic dependent launch.  A kernel launched with launch_pdl() lets the next such
// kernel on the stream start its prologue (CTA launch, barrier set-up, TMEM allocation)
// while this one finishes; every global-memory access of the next kernel comes after its
// pdl_wait(), which returns once the previous grid has completed and its writes are
// visible, so stream order is kept for data.
__device__ __forceinline__ void pdl_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                       Args &&...args) {
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
    return cudaLaunchKernelEx(&cfg, kern, static_cast<Args &&>(args)...);
}

// Workspace of the weight-stationary matvecs (fp16 and Q8_0): a status word in a 256-byte
// header (split-K partial sums are reduced in distributed shared memory, not here).
constexpr size_t kWsHeaderBytes = 256;
constexpr unsigned kWsStatusTimeout = 1u;

// Named barrier over `nthreads` threads (a subset of the CTA).
__device__ __forceinline__ void named_bar_sync(int id, int nthreads) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

__device__ __forceinline__ unsigned ld_acquire_u32(const unsigned *p) {
    unsigned v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ unsigned long long ld_relaxed_u64(const unsigned long long *p) {
    unsigned long long v;
    asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ void red_release_add_u32(unsigned *p, unsigned v) {
    asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// Read-only 16-byte global load that does not allocate in L1.
__device__ __forceinline__ uint4 ldg_nc_v4(const void *p) {
    uint4 r;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "l"(p));
    return r;
}

// Order-preserving map of an fp32 value to uint32 (-0 is first folded onto +0, so
// equal values map to equal codes).  Larger float -> larger code.
__device__ __forceinline__ uint32_t float_order_code(float x) {
    uint32_t u = __float_as_uint(x + 0.0f);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// (value desc, index asc) as one 64-bit key: max over keys = greedy argmax with the
// lowest-index tie-break.  Every finite or infinite logit gives a key > 0.
__device__ __forceinline__ unsigned long long argmax_key(float logit, uint32_t index) {
    return (static_cast<unsigned long long>(float_order_code(logit)) << 32) |
           static_cast<unsigned long long>(0xffffffffu - index);
}

__device__ __forceinline__ uint32_t argmax_key_index(unsigned long long key) {
    return 0xffffffffu - static_cast<uint32_t>(key & 0xffffffffull);
}

// Warp-wide max of 64-bit keys with two 32-bit redux.sync reductions: the max high word,
// then the max low word among the lanes holding it.  All 32 lanes must take part.
__device__ __forceinline__ unsigned long long warp_max_u64(unsigned long long v) {
    const unsigned hi = static_cast<unsigned>(v >> 32);
    const unsigned mh = __reduce_max_sync(0xffffffffu, hi);
    const unsigned ml = __reduce_max_sync(0xffffffffu, hi == mh ? static_cast<unsigned>(v) : 0u);
    return (static_cast<unsigned long long>(mh) << 32) | ml;
}

}  // namespace dspark
