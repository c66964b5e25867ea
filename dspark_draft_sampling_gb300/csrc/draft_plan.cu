// Draft step with the base logits produced on the device: lm_head matvec -> Markov draft,
// recorded into one CUDA graph.
//
// vllm.cpp issue #436 ("W7 LANDED") leaves open "the device-returning block-forward
// variant": the base logits [num_reqs, k, draft_vocab] are downloaded to the host after the
// backbone.  Here the draft head's projection (SharpInference issue #441, "Observation":
// the lm_head is one of the M = B small-M fp16 GEMMs) writes them straight into device
// memory with the weight-stationary matvec, and the Markov kernel consumes them there;
// both are captured in one graph, so a draft step is one graph launch and the only
// device -> host traffic is the caller's read of out_ids.
#include <new>

#include "markov.cuh"

struct dspark_draft_plan {
    cudaGraph_t graph;
    cudaGraphExec_t exec;
};

extern "C" dspark_status dspark_draft_plan_create(const uint16_t *lm_head, const uint16_t *hidden_states,
                                                  int hidden_dim, const uint16_t *markov_w1,
                                                  const uint16_t *markov_w2, const int32_t *d2t, int64_t *prev,
                                                  int num_reqs, int k, int vocab, int rank, float *base_logits,
                                                  int64_t *out_ids, void *markov_workspace,
                                                  size_t markov_workspace_bytes, void *ws_workspace,
                                                  size_t ws_workspace_bytes, dspark_draft_plan **plan_out) {
    using namespace dspark;
    clear_error();
    if (!plan_out) return fail(DSPARK_ERR_INVALID, "draft_plan_create: null plan_out");
    *plan_out = nullptr;
    if (num_reqs < 1 || k < 1 || vocab < 1 || hidden_dim < 8)
        return fail(DSPARK_ERR_INVALID, "draft_plan_create: bad sizes num_reqs=%d k=%d vocab=%d hidden=%d", num_reqs,
                    k, vocab, hidden_dim);
    if (num_reqs * k > 16)
        return fail(DSPARK_ERR_UNSUPPORTED, "draft_plan_create: num_reqs * k = %d > 16 matvec rows", num_reqs * k);
    if (!lm_head || !hidden_states || !base_logits)
        return fail(DSPARK_ERR_INVALID, "draft_plan_create: null pointer argument");
    cudaStream_t s = nullptr;
    cudaError_t e = cudaStreamCreateWithFlags(&s, cudaStreamNonBlocking);
    if (e != cudaSuccess) return cuda_fail(e, "cudaStreamCreateWithFlags");
    e = cudaStreamBeginCapture(s, cudaStreamCaptureModeThreadLocal);
    if (e != cudaSuccess) {
        cudaStreamDestroy(s);
        return cuda_fail(e, "cudaStreamBeginCapture");
    }
    // base[r, i, :] = lm_head . hidden[r * k + i, :]  (fp32 out: [num_reqs * k, vocab] = [num_reqs, k, vocab])
    dspark_status st = dspark_ws_matvec(lm_head, hidden_states, base_logits, 1, num_reqs * k, vocab, hidden_dim,
                                        ws_workspace, ws_workspace_bytes, reinterpret_cast<dspark_stream_t>(s));
    if (st == DSPARK_OK)
        st = markov_enqueue(base_logits, markov_w1, markov_w2, d2t, prev, num_reqs, k, vocab, rank, out_ids, nullptr,
                            nullptr, markov_workspace, markov_workspace_bytes, 0u, kDefaultTimeoutNs, s);
    cudaGraph_t graph = nullptr;
    e = cudaStreamEndCapture(s, &graph);
    cudaStreamDestroy(s);
    if (st != DSPARK_OK) {
        if (graph) cudaGraphDestroy(graph);
        return st;
    }
    if (e != cudaSuccess) return cuda_fail(e, "cudaStreamEndCapture");
    cudaGraphExec_t exec = nullptr;
    e = cudaGraphInstantiate(&exec, graph, 0);
    if (e != cudaSuccess) {
        cudaGraphDestroy(graph);
        return cuda_fail(e, "cudaGraphInstantiate");
    }
    auto *plan = new (std::nothrow) dspark_draft_plan{graph, exec};
    if (!plan) {
        cudaGraphExecDestroy(exec);
        cudaGraphDestroy(graph);
        return fail(DSPARK_ERR_CUDA, "draft_plan_create: out of host memory");
    }
    *plan_out = plan;
    return DSPARK_OK;
}

extern "C" dspark_status dspark_draft_plan_launch(dspark_draft_plan *plan, dspark_stream_t stream) {
    dspark::clear_error();
    if (!plan) return dspark::fail(DSPARK_ERR_INVALID, "draft_plan_launch: null plan");
    cudaError_t e = cudaGraphLaunch(plan->exec, reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return dspark::cuda_fail(e, "cudaGraphLaunch");
    return DSPARK_OK;
}

extern "C" void dspark_draft_plan_destroy(dspark_draft_plan *plan) {
    if (!plan) return;
    cudaGraphExecDestroy(plan->exec);
    cudaGraphDestroy(plan->graph);
    delete plan;
}
