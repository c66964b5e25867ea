// Markov block-draft sampler: host side of the C ABI (argument checks, workspace,
// launch, graph plan, status word, allocation-free variant).  The kernel itself is the
// tcgen05 form in markov_tc.cu: all k draft positions in one persistent cooperative launch.
//
// Method (vllm.cpp issue #436 "SPEC-DSPARK W7", section "The fix"): per position,
// gather markov_w1[prev], bias GEMV over the whole bf16 markov_w2 [vocab, rank], add the
// position's base-logit row, greedy argmax with lowest-index tie-break, d2t map, and
// carry prev on the device; only the final [num_reqs, k] ids leave the GPU.
#include <cuda.h>

#include <mutex>
#include <new>

#include "markov.cuh"

namespace dspark {

size_t workspace_bytes(int k) {
    const size_t keys = size_t(k > 0 ? k : 0) * kMaxReqs * sizeof(unsigned long long);
    return (kHeaderBytes + keys + 255) / 256 * 256;
}

dspark_status markov_enqueue(const float *base, const uint16_t *w1, const uint16_t *w2, const int32_t *d2t,
                             int64_t *prev, int B, int k, int V, int R, int64_t *out_ids, float *dbg_logits,
                             float *dbg_bias, void *workspace, size_t ws_bytes, unsigned bar_extra,
                             unsigned long long timeout_ns, cudaStream_t stream, bool clear_out_ids, int kernel) {
    clear_error();
    if (kernel != kMarkovAuto && kernel != kMarkovGrid && kernel != kMarkovCluster)
        return fail(DSPARK_ERR_INVALID, "markov: kernel %d", kernel);
    if (B < 0 || k < 0 || V < 1 || R < 1) return fail(DSPARK_ERR_INVALID, "markov: bad sizes B=%d k=%d V=%d R=%d", B, k, V, R);
    if (R != 64 && R != 128 && R != 256)
        return fail(DSPARK_ERR_UNSUPPORTED, "markov: rank %d not in {64, 128, 256}", R);
    if (B > kMaxReqs) return fail(DSPARK_ERR_UNSUPPORTED, "markov: num_reqs %d > %d", B, kMaxReqs);
    if (B == 0 || k == 0) return DSPARK_OK;  // nothing to enqueue
    if (!base || !w1 || !w2 || !prev || !out_ids || !workspace)
        return fail(DSPARK_ERR_INVALID, "markov: null pointer argument");
    if (!aligned(w1, 16) || !aligned(w2, 16))
        return fail(DSPARK_ERR_INVALID, "markov: markov_w1/markov_w2 must be 16-byte aligned");
    if (!aligned(base, 4) || !aligned(prev, 8) || !aligned(out_ids, 8) || (d2t && !aligned(d2t, 4)) ||
        (dbg_logits && !aligned(dbg_logits, 4)) || (dbg_bias && !aligned(dbg_bias, 4)))
        return fail(DSPARK_ERR_INVALID, "markov: misaligned tensor pointer");
    if (!aligned(workspace, 256)) return fail(DSPARK_ERR_INVALID, "markov: workspace must be 256-byte aligned");
    if (ws_bytes < workspace_bytes(k))
        return fail(DSPARK_ERR_INVALID, "markov: workspace of %zu bytes < required %zu", ws_bytes, workspace_bytes(k));
    int sms = 0;
    int rc = current_sm_count(&sms);
    if (rc != DSPARK_OK) return static_cast<dspark_status>(rc);

    int C = 0;  // cluster size of the single-cluster form, 0 for the grid form
    if (kernel == kMarkovCluster || (kernel == kMarkovAuto && markov_auto_kernel(base, B, V, R, k) == kMarkovCluster)) {
        if (aligned(base, 16)) C = markov_cluster_size(B, V, R, k);
        if (kernel == kMarkovCluster && C == 0)
            return fail(DSPARK_ERR_UNSUPPORTED,
                        "markov: the single-cluster kernel does not apply (vocab %d, rank %d, k %d; vocab a "
                        "multiple of 4, base 16-byte aligned, markov_w1 + markov_w2 in one cluster)",
                        V, R, k);
    }

    unsigned char *ws = static_cast<unsigned char *>(workspace);
    cudaError_t e;
    if (clear_out_ids) {  // every id -1 until the kernel writes it
        e = cudaMemsetAsync(out_ids, 0xFF, size_t(B) * size_t(k) * sizeof(int64_t), stream);
        if (e != cudaSuccess) return cuda_fail(e, "cudaMemsetAsync(out_ids)");
    }
    if (C == 0) {  // the grid form's barrier counter and keys start from zero
        e = cudaMemsetAsync(ws, 0, workspace_bytes(k), stream);
        if (e != cudaSuccess) return cuda_fail(e, "cudaMemsetAsync(markov workspace)");
    }
    MarkovArgs args;
    args.base = base;
    args.w1 = w1;
    args.w2 = w2;
    args.d2t = d2t;
    args.prev = prev;
    args.out_ids = out_ids;
    args.dbg_logits = dbg_logits;
    args.dbg_bias = dbg_bias;
    args.bar_count = reinterpret_cast<unsigned *>(ws);
    args.status = reinterpret_cast<unsigned *>(ws) + 1;
    args.best = reinterpret_cast<unsigned long long *>(ws + kHeaderBytes);
    args.B = B;
    args.k = k;
    args.V = V;
    args.bar_extra = bar_extra;
    args.timeout_ns = timeout_ns;
    if (C > 0) return launch_markov_cluster(args, R, C, stream);
    return launch_markov_tc(args, R, markov_grid(V, sms), stream);
}

int markov_auto_kernel(const float *base, int B, int V, int R, int k) {
    // The single-cluster exchange sends every request's key and candidate row to every CTA
    // of the cluster; beyond two requests that volume costs more per position than the grid
    // form's global round trips save (measured on GB300).  Both kernels give the same bits.
    return (B <= kMarkovClusterAutoMaxReqs && aligned(base, 16) && markov_cluster_size(B, V, R, k) > 0)
               ? kMarkovCluster
               : kMarkovGrid;
}

}  // namespace dspark

struct dspark_markov_plan {
    cudaGraph_t graph;
    cudaGraphExec_t exec;
};

extern "C" size_t dspark_markov_workspace_bytes(int num_reqs, int k, int vocab, int rank) {
    (void)num_reqs;
    (void)vocab;
    (void)rank;
    return dspark::workspace_bytes(k);
}

extern "C" dspark_status dspark_markov_draft(const float *base_logits, const uint16_t *markov_w1,
                                             const uint16_t *markov_w2, const int32_t *d2t, int64_t *prev,
                                             int num_reqs, int k, int vocab, int rank, int64_t *out_ids,
                                             float *dbg_logits, float *dbg_bias, void *workspace,
                                             size_t workspace_bytes, dspark_stream_t stream) {
    return dspark::markov_enqueue(base_logits, markov_w1, markov_w2, d2t, prev, num_reqs, k, vocab, rank, out_ids,
                                  dbg_logits, dbg_bias, workspace, workspace_bytes, 0u, dspark::kDefaultTimeoutNs,
                                  reinterpret_cast<cudaStream_t>(stream));
}

extern "C" dspark_status dspark_markov_draft_kernel(const float *base_logits, const uint16_t *markov_w1,
                                                    const uint16_t *markov_w2, const int32_t *d2t, int64_t *prev,
                                                    int num_reqs, int k, int vocab, int rank, int64_t *out_ids,
                                                    float *dbg_logits, float *dbg_bias, void *workspace,
                                                    size_t workspace_bytes, int kernel, dspark_stream_t stream) {
    return dspark::markov_enqueue(base_logits, markov_w1, markov_w2, d2t, prev, num_reqs, k, vocab, rank, out_ids,
                                  dbg_logits, dbg_bias, workspace, workspace_bytes, 0u, dspark::kDefaultTimeoutNs,
                                  reinterpret_cast<cudaStream_t>(stream), false, kernel);
}

extern "C" int dspark_markov_kernel_for(int num_reqs, int k, int vocab, int rank) {
    if (k < 1 || vocab < 1) return dspark::kMarkovGrid;
    // an aligned stand-in for the base pointer: the choice is made for a 16-byte aligned base
    return dspark::markov_auto_kernel(reinterpret_cast<const float *>(uintptr_t(256)), num_reqs, vocab, rank, k);
}

extern "C" dspark_status dspark_markov_draft_debug(const float *base_logits, const uint16_t *markov_w1,
                                                   const uint16_t *markov_w2, const int32_t *d2t, int64_t *prev,
                                                   int num_reqs, int k, int vocab, int rank, int64_t *out_ids,
                                                   void *workspace, size_t workspace_bytes,
                                                   unsigned missing_arrivals, unsigned timeout_us,
                                                   dspark_stream_t stream) {
    if (timeout_us == 0 || timeout_us > 10u * 1000u * 1000u)
        return dspark::fail(DSPARK_ERR_INVALID, "markov_debug: timeout_us must be in [1, 10^7]");
    return dspark::markov_enqueue(base_logits, markov_w1, markov_w2, d2t, prev, num_reqs, k, vocab, rank, out_ids,
                                  nullptr, nullptr, workspace, workspace_bytes, missing_arrivals,
                                  static_cast<unsigned long long>(timeout_us) * 1000ull,
                                  reinterpret_cast<cudaStream_t>(stream), false, dspark::kMarkovGrid);
}

// ---- allocation-free variant ----------------------------------------------------------
// Scratch for dspark_markov_draft_noalloc: the same header + per-position argmax keys that
// a caller-provided workspace holds, sized for at most kNoAllocMaxK positions.  It lives in
// the library's own device memory, allocated when the module is loaded on a device and
// held until the process exits.  In host code `g_markov_noalloc_scratch` is only a host-side
// handle for the symbol: its device address comes from cudaGetSymbolAddress below.
namespace dspark {
namespace {
constexpr int kNoAllocMaxK = 64;
constexpr size_t kNoAllocScratchBytes = kHeaderBytes + size_t(kNoAllocMaxK) * kMaxReqs * sizeof(unsigned long long);
static_assert(kNoAllocScratchBytes == 4352, "scratch size");
}  // namespace
}  // namespace dspark

static __device__ __align__(256) unsigned char g_markov_noalloc_scratch[dspark::kNoAllocScratchBytes];

namespace dspark {
namespace {
using PFN_ctx_get_current = CUresult (*)(CUcontext *);
using PFN_ctx_get_id = CUresult (*)(CUcontext, unsigned long long *);

// Process-unique id of the calling thread's current CUDA context (0 if none is current
// or the driver does not provide the query).  Ids are never reused, unlike context handles.
unsigned long long current_context_id() {
    static PFN_ctx_get_current get_current = nullptr;
    static PFN_ctx_get_id get_id = nullptr;
    static bool looked_up = false;
    if (!looked_up) {
        void *f1 = nullptr, *f2 = nullptr;
        cudaDriverEntryPointQueryResult q1 = cudaDriverEntryPointSymbolNotFound, q2 = q1;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f1, 12000, cudaEnableDefault, &q1) == cudaSuccess &&
            q1 == cudaDriverEntryPointSuccess)
            get_current = reinterpret_cast<PFN_ctx_get_current>(f1);
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &f2, 12000, cudaEnableDefault, &q2) == cudaSuccess &&
            q2 == cudaDriverEntryPointSuccess)
            get_id = reinterpret_cast<PFN_ctx_get_id>(f2);
        looked_up = true;
    }
    if (!get_current || !get_id) return 0;
    CUcontext ctx = nullptr;
    unsigned long long id = 0;
    if (get_current(&ctx) != CUDA_SUCCESS || !ctx || get_id(ctx, &id) != CUDA_SUCCESS) return 0;
    return id;
}

// Device address of the scratch array in the current context.  It is looked up with
// cudaGetSymbolAddress the first time a context uses the entry point (once per device in the
// usual one-context-per-device process) and cached with that context's id; a different
// context on the same device (a context the caller created, or the primary context again
// after cudaDeviceReset) has its own copy of the array and gets its own lookup.
dspark_status noalloc_scratch(void **out) {
    struct Entry {
        unsigned long long ctx_id;
        void *addr;
    };
    static Entry cache[64] = {};
    static std::mutex mu;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    if (dev < 0 || dev >= 64) return fail(DSPARK_ERR_UNSUPPORTED, "markov_noalloc: device ordinal %d >= 64", dev);
    const unsigned long long id = current_context_id();
    std::lock_guard<std::mutex> lock(mu);
    if (id != 0 && cache[dev].ctx_id == id && cache[dev].addr) {
        *out = cache[dev].addr;
        return DSPARK_OK;
    }
    void *p = nullptr;
    e = cudaGetSymbolAddress(&p, g_markov_noalloc_scratch);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(markov scratch)");
    // the lookup makes the runtime's context current if none was: key the cache on it
    cache[dev].ctx_id = id != 0 ? id : current_context_id();
    cache[dev].addr = p;
    *out = p;
    return DSPARK_OK;
}
}  // namespace
}  // namespace dspark

extern "C" dspark_status dspark_markov_draft_noalloc(const float *base_logits, const uint16_t *markov_w1,
                                                     const uint16_t *markov_w2, const int32_t *d2t, int64_t *prev,
                                                     int num_reqs, int k, int vocab, int rank, int64_t *out_ids,
                                                     dspark_stream_t stream) {
    dspark::clear_error();
    if (k > dspark::kNoAllocMaxK)
        return dspark::fail(DSPARK_ERR_UNSUPPORTED,
                            "markov_noalloc: k=%d exceeds the %d positions its static scratch holds; "
                            "use dspark_markov_draft with a workspace",
                            k, dspark::kNoAllocMaxK);
    void *scratch = nullptr;
    dspark_status st = dspark::noalloc_scratch(&scratch);
    if (st != DSPARK_OK) return st;
    // out_ids is set to -1 first: the status word in the static scratch cannot be read by the
    // caller, so a position the kernel could not finish (a device-side wait that gave up)
    // shows as -1 instead of a stale id
    return dspark::markov_enqueue(base_logits, markov_w1, markov_w2, d2t, prev, num_reqs, k, vocab, rank, out_ids,
                                  nullptr, nullptr, scratch, dspark::kNoAllocScratchBytes, 0u,
                                  dspark::kDefaultTimeoutNs, reinterpret_cast<cudaStream_t>(stream), true);
}

extern "C" dspark_status dspark_markov_status(const void *workspace, dspark_stream_t stream) {
    dspark::clear_error();
    if (!workspace) return dspark::fail(DSPARK_ERR_INVALID, "markov_status: null workspace");
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    cudaError_t e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return dspark::cuda_fail(e, "cudaStreamSynchronize");
    unsigned st = 0;
    e = cudaMemcpy(&st, static_cast<const unsigned *>(workspace) + 1, sizeof st, cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return dspark::cuda_fail(e, "cudaMemcpy(markov status)");
    if (st & dspark::kStatusTimeout) return dspark::fail(DSPARK_ERR_TIMEOUT, "markov: a device-side wait timed out");
    if (st & dspark::kStatusIndex)
        return dspark::fail(DSPARK_ERR_INDEX, "markov: a prev or d2t entry was out of range");
    return DSPARK_OK;
}

extern "C" dspark_status dspark_markov_plan_create(const float *base_logits, const uint16_t *markov_w1,
                                                   const uint16_t *markov_w2, const int32_t *d2t, int64_t *prev,
                                                   int num_reqs, int k, int vocab, int rank, int64_t *out_ids,
                                                   void *workspace, size_t workspace_bytes,
                                                   dspark_markov_plan **plan_out) {
    dspark::clear_error();
    if (!plan_out) return dspark::fail(DSPARK_ERR_INVALID, "markov_plan_create: null plan_out");
    *plan_out = nullptr;
    cudaStream_t s = nullptr;
    cudaError_t e = cudaStreamCreateWithFlags(&s, cudaStreamNonBlocking);
    if (e != cudaSuccess) return dspark::cuda_fail(e, "cudaStreamCreateWithFlags");
    e = cudaStreamBeginCapture(s, cudaStreamCaptureModeThreadLocal);
    if (e != cudaSuccess) {
        cudaStreamDestroy(s);
        return dspark::cuda_fail(e, "cudaStreamBeginCapture");
    }
    dspark_status st = dspark::markov_enqueue(base_logits, markov_w1, markov_w2, d2t, prev, num_reqs, k, vocab, rank,
                                              out_ids, nullptr, nullptr, workspace, workspace_bytes, 0u,
                                              dspark::kDefaultTimeoutNs, s);
    cudaGraph_t graph = nullptr;
    e = cudaStreamEndCapture(s, &graph);
    cudaStreamDestroy(s);
    if (st != DSPARK_OK) {
        if (graph) cudaGraphDestroy(graph);
        return st;
    }
    if (e != cudaSuccess) return dspark::cuda_fail(e, "cudaStreamEndCapture");
    cudaGraphExec_t exec = nullptr;
    e = cudaGraphInstantiate(&exec, graph, 0);
    if (e != cudaSuccess) {
        cudaGraphDestroy(graph);
        return dspark::cuda_fail(e, "cudaGraphInstantiate");
    }
    auto *plan = new (std::nothrow) dspark_markov_plan{graph, exec};
    if (!plan) {
        cudaGraphExecDestroy(exec);
        cudaGraphDestroy(graph);
        return dspark::fail(DSPARK_ERR_CUDA, "markov_plan_create: out of host memory");
    }
    *plan_out = plan;
    return DSPARK_OK;
}

extern "C" dspark_status dspark_markov_plan_launch(dspark_markov_plan *plan, dspark_stream_t stream) {
    dspark::clear_error();
    if (!plan) return dspark::fail(DSPARK_ERR_INVALID, "markov_plan_launch: null plan");
    cudaError_t e = cudaGraphLaunch(plan->exec, reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return dspark::cuda_fail(e, "cudaGraphLaunch");
    return DSPARK_OK;
}

extern "C" void dspark_markov_plan_destroy(dspark_markov_plan *plan) {
    if (!plan) return;
    cudaGraphExecDestroy(plan->exec);
    cudaGraphDestroy(plan->graph);
    delete plan;
}
