// Confidence-gated draft: the probe decides on the device whether the Markov draft runs.
//
// ds4 PR #772 ("Summary", "Root cause") moves the proposer's confidence gate to the GPU but
// still reads its 4-byte decision back to the host before drafting continues.  Here the
// decision never leaves the device: one CUDA graph holds the probe kernel and a conditional
// IF node whose body is the k-position Markov draft; the probe kernel sets the node's
// condition with cudaGraphSetConditional, so the draft runs (or is skipped) without a host
// round trip.  The gate is still written to gate_out for the caller's bookkeeping.
#include <new>

#include "markov.cuh"

struct dspark_gated_plan {
    cudaGraph_t graph;
    cudaGraphExec_t exec;
};

extern "C" dspark_status dspark_gated_draft_plan_create(
    const void *w_q8_0, const float *probe_input, int K, float bias, float threshold, float *logit_out,
    int32_t *gate_out, const float *base_logits, const uint16_t *markov_w1, const uint16_t *markov_w2,
    const int32_t *d2t, int64_t *prev, int num_reqs, int k, int vocab, int rank, int64_t *out_ids,
    void *workspace, size_t workspace_bytes, dspark_gated_plan **plan_out) {
    using namespace dspark;
    clear_error();
    if (!plan_out) return fail(DSPARK_ERR_INVALID, "gated_draft_plan_create: null plan_out");
    *plan_out = nullptr;
    if (K <= 0 || (K % 32) != 0) return fail(DSPARK_ERR_INVALID, "gated_draft_plan_create: K=%d", K);
    if (num_reqs < 1 || k < 1) return fail(DSPARK_ERR_INVALID, "gated_draft_plan_create: empty draft");

    cudaGraph_t graph = nullptr;
    cudaError_t e = cudaGraphCreate(&graph, 0);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGraphCreate");
    cudaStream_t s = nullptr;
    dspark_status st = DSPARK_OK;
    auto bail = [&](dspark_status code) {
        if (s) cudaStreamDestroy(s);
        cudaGraphDestroy(graph);
        return code;
    };
    cudaGraphConditionalHandle cond = 0;
    e = cudaGraphConditionalHandleCreate(&cond, graph, 0, cudaGraphCondAssignDefault);
    if (e != cudaSuccess) return bail(cuda_fail(e, "cudaGraphConditionalHandleCreate"));
    e = cudaStreamCreateWithFlags(&s, cudaStreamNonBlocking);
    if (e != cudaSuccess) return bail(cuda_fail(e, "cudaStreamCreateWithFlags"));

    // 1) the probe (one probe; it sets the condition)
    e = cudaStreamBeginCaptureToGraph(s, graph, nullptr, nullptr, 0, cudaStreamCaptureModeThreadLocal);
    if (e != cudaSuccess) return bail(cuda_fail(e, "cudaStreamBeginCaptureToGraph(probe)"));
    st = probe_enqueue(w_q8_0, probe_input, K, K, nullptr, 0, 0, bias, threshold, 1, logit_out, gate_out, s, cond, 1);
    cudaGraph_t captured = nullptr;
    e = cudaStreamEndCapture(s, &captured);
    if (st != DSPARK_OK) return bail(st);
    if (e != cudaSuccess) return bail(cuda_fail(e, "cudaStreamEndCapture(probe)"));
    cudaGraphNode_t probe_node = nullptr;
    size_t nnodes = 1;
    e = cudaGraphGetNodes(graph, &probe_node, &nnodes);
    if (e != cudaSuccess || nnodes != 1) return bail(fail(DSPARK_ERR_CUDA, "gated_draft_plan_create: probe capture"));

    // 2) IF node after the probe; its body is the Markov draft
    cudaGraphNodeParams cp = {};
    cp.type = cudaGraphNodeTypeConditional;
    cp.conditional.handle = cond;
    cp.conditional.type = cudaGraphCondTypeIf;
    cp.conditional.size = 1;
    cudaGraphNode_t cond_node = nullptr;
    e = cudaGraphAddNode(&cond_node, graph, &probe_node, nullptr, 1, &cp);
    if (e != cudaSuccess) return bail(cuda_fail(e, "cudaGraphAddNode(conditional)"));
    cudaGraph_t body = cp.conditional.phGraph_out[0];
    e = cudaStreamBeginCaptureToGraph(s, body, nullptr, nullptr, 0, cudaStreamCaptureModeThreadLocal);
    if (e != cudaSuccess) return bail(cuda_fail(e, "cudaStreamBeginCaptureToGraph(draft)"));
    st = markov_enqueue(base_logits, markov_w1, markov_w2, d2t, prev, num_reqs, k, vocab, rank, out_ids, nullptr,
                        nullptr, workspace, workspace_bytes, 0u, kDefaultTimeoutNs, s);
    e = cudaStreamEndCapture(s, &captured);
    if (st != DSPARK_OK) return bail(st);
    if (e != cudaSuccess) return bail(cuda_fail(e, "cudaStreamEndCapture(draft)"));
    cudaStreamDestroy(s);
    s = nullptr;

    cudaGraphExec_t exec = nullptr;
    e = cudaGraphInstantiate(&exec, graph, 0);
    if (e != cudaSuccess) return bail(cuda_fail(e, "cudaGraphInstantiate(gated draft)"));
    auto *plan = new (std::nothrow) dspark_gated_plan{graph, exec};
    if (!plan) {
        cudaGraphExecDestroy(exec);
        return bail(fail(DSPARK_ERR_CUDA, "gated_draft_plan_create: out of host memory"));
    }
    *plan_out = plan;
    return DSPARK_OK;
}

extern "C" dspark_status dspark_gated_draft_plan_launch(dspark_gated_plan *plan, dspark_stream_t stream) {
    dspark::clear_error();
    if (!plan) return dspark::fail(DSPARK_ERR_INVALID, "gated_draft_plan_launch: null plan");
    cudaError_t e = cudaGraphLaunch(plan->exec, reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return dspark::cuda_fail(e, "cudaGraphLaunch");
    return DSPARK_OK;
}

extern "C" void dspark_gated_draft_plan_destroy(dspark_gated_plan *plan) {
    if (!plan) return;
    cudaGraphExecDestroy(plan->exec);
    cudaGraphDestroy(plan->graph);
    delete plan;
}
