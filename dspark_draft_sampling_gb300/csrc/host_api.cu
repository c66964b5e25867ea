// Host-buffer forms of the three draft-step operations.
//
// Each takes its per-call inputs in host memory and returns its outputs to host memory: the
// host-to-device copies, the same kernel as the device-pointer form, and the device-to-host
// copies are enqueued in that order on the caller's stream, so a cycle that starts from host
// data needs one call per operation and one stream synchronization.  Resident tensors
// (markov_w1/w2, d2t, the probe's Q8_0 row, the projection weights) stay device pointers.
// Host buffers should be page-locked (cudaHostAlloc / cudaHostRegister) for the copies to
// run asynchronously; with pageable memory they still work but block the calling thread.
// Pinned host-to-device copies queued on several streams are served in the order they become
// ready, not interleaved, so a caller that overlaps two operations can record the optional
// inputs_copied event of the first and make the second's stream wait on it: the small,
// urgent input then never queues behind a large one.
#include "markov.cuh"

namespace {

size_t up256(size_t x) { return (x + 255) & ~size_t(255); }

// Record the caller's optional event once the inputs are on the device.
dspark_status mark_copied(void *event, cudaStream_t s) {
    if (!event) return DSPARK_OK;
    const cudaError_t e = cudaEventRecord(static_cast<cudaEvent_t>(event), s);
    if (e != cudaSuccess) return dspark::cuda_fail(e, "inputs_copied event");
    return DSPARK_OK;
}

dspark_status copy(void *dst, const void *src, size_t bytes, cudaMemcpyKind kind, cudaStream_t s, const char *what) {
    if (bytes == 0) return DSPARK_OK;
    const cudaError_t e = cudaMemcpyAsync(dst, src, bytes, kind, s);
    if (e != cudaSuccess) return dspark::cuda_fail(e, what);
    return DSPARK_OK;
}

}  // namespace

extern "C" size_t dspark_markov_draft_host_scratch_bytes(int num_reqs, int k, int vocab, int rank) {
    if (num_reqs < 0 || k < 0 || vocab < 1) return 0;
    const size_t B = static_cast<size_t>(num_reqs), K = static_cast<size_t>(k), V = static_cast<size_t>(vocab);
    return up256(B * K * V * 4) + up256(B * 8) + up256(B * K * 8) + dspark_markov_workspace_bytes(num_reqs, k, vocab, rank);
}

extern "C" dspark_status dspark_markov_draft_host(const float *base_host, const uint16_t *markov_w1,
                                                  const uint16_t *markov_w2, const int32_t *d2t, int64_t *prev_host,
                                                  int num_reqs, int k, int vocab, int rank, int64_t *out_ids_host,
                                                  void *device_scratch, size_t scratch_bytes, void *inputs_copied,
                                                  dspark_stream_t stream) {
    using namespace dspark;
    clear_error();
    if (num_reqs < 0 || k < 0 || vocab < 1 || rank < 1)
        return fail(DSPARK_ERR_INVALID, "markov_draft_host: bad sizes B=%d k=%d V=%d R=%d", num_reqs, k, vocab, rank);
    if (rank != 64 && rank != 128 && rank != 256)
        return fail(DSPARK_ERR_UNSUPPORTED, "markov_draft_host: rank %d not in {64, 128, 256}", rank);
    if (num_reqs > kMaxReqs) return fail(DSPARK_ERR_UNSUPPORTED, "markov_draft_host: num_reqs %d > %d", num_reqs, kMaxReqs);
    if (num_reqs == 0 || k == 0) return DSPARK_OK;  // nothing to enqueue
    if (!base_host || !markov_w1 || !markov_w2 || !prev_host || !out_ids_host || !device_scratch)
        return fail(DSPARK_ERR_INVALID, "markov_draft_host: null pointer argument");
    if (!aligned(markov_w1, 16) || !aligned(markov_w2, 16) || !aligned(device_scratch, 256))
        return fail(DSPARK_ERR_INVALID, "markov_draft_host: markov_w1/w2 must be 16-byte and scratch 256-byte aligned");
    const size_t need = dspark_markov_draft_host_scratch_bytes(num_reqs, k, vocab, rank);
    if (scratch_bytes < need)
        return fail(DSPARK_ERR_INVALID, "markov_draft_host: scratch of %zu bytes < required %zu", scratch_bytes, need);
    const size_t B = static_cast<size_t>(num_reqs), K = static_cast<size_t>(k), V = static_cast<size_t>(vocab);
    unsigned char *p = static_cast<unsigned char *>(device_scratch);
    float *base_d = reinterpret_cast<float *>(p);
    p += up256(B * K * V * 4);
    int64_t *prev_d = reinterpret_cast<int64_t *>(p);
    p += up256(B * 8);
    int64_t *out_d = reinterpret_cast<int64_t *>(p);
    p += up256(B * K * 8);
    const size_t ws_bytes = dspark_markov_workspace_bytes(num_reqs, k, vocab, rank);
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    dspark_status st = copy(base_d, base_host, B * K * V * 4, cudaMemcpyHostToDevice, s, "markov_draft_host: base copy");
    if (st == DSPARK_OK) st = copy(prev_d, prev_host, B * 8, cudaMemcpyHostToDevice, s, "markov_draft_host: prev copy");
    if (st == DSPARK_OK) st = mark_copied(inputs_copied, s);
    if (st == DSPARK_OK)
        st = dspark_markov_draft(base_d, markov_w1, markov_w2, d2t, prev_d, num_reqs, k, vocab, rank, out_d, nullptr,
                                 nullptr, p, ws_bytes, stream);
    if (st == DSPARK_OK) st = copy(out_ids_host, out_d, B * K * 8, cudaMemcpyDeviceToHost, s, "markov_draft_host: ids copy");
    if (st == DSPARK_OK) st = copy(prev_host, prev_d, B * 8, cudaMemcpyDeviceToHost, s, "markov_draft_host: prev copy");
    return st;
}

extern "C" size_t dspark_conf_probe_host_scratch_bytes(int K, int n_probes) {
    if (K < 0 || n_probes < 0) return 0;
    const size_t n = static_cast<size_t>(n_probes);
    return up256(n * static_cast<size_t>(K) * 4) + 2 * up256(n * 4);
}

extern "C" dspark_status dspark_conf_probe_host(const void *w_q8_0, const float *hidden_host, float bias,
                                                float threshold, int K, int n_probes, float *logit_host,
                                                int32_t *gate_host, void *device_scratch, size_t scratch_bytes,
                                                void *inputs_copied, dspark_stream_t stream) {
    using namespace dspark;
    clear_error();
    if (K <= 0 || (K % 32) != 0 || n_probes < 0)
        return fail(DSPARK_ERR_INVALID, "conf_probe_host: bad sizes K=%d n=%d", K, n_probes);
    if (!(threshold > 0.f && threshold < 1.f))
        return fail(DSPARK_ERR_INVALID, "conf_probe_host: threshold must lie in (0, 1)");
    if (n_probes == 0) return DSPARK_OK;
    if (!w_q8_0 || !hidden_host || !gate_host || !device_scratch)
        return fail(DSPARK_ERR_INVALID, "conf_probe_host: null pointer argument");
    if (!aligned(device_scratch, 256)) return fail(DSPARK_ERR_INVALID, "conf_probe_host: scratch must be 256-byte aligned");
    const size_t need = dspark_conf_probe_host_scratch_bytes(K, n_probes);
    if (scratch_bytes < need)
        return fail(DSPARK_ERR_INVALID, "conf_probe_host: scratch of %zu bytes < required %zu", scratch_bytes, need);
    const size_t n = static_cast<size_t>(n_probes);
    unsigned char *p = static_cast<unsigned char *>(device_scratch);
    float *hid_d = reinterpret_cast<float *>(p);
    p += up256(n * static_cast<size_t>(K) * 4);
    float *logit_d = reinterpret_cast<float *>(p);
    p += up256(n * 4);
    int32_t *gate_d = reinterpret_cast<int32_t *>(p);
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    dspark_status st = copy(hid_d, hidden_host, n * static_cast<size_t>(K) * 4, cudaMemcpyHostToDevice, s,
                            "conf_probe_host: hidden copy");
    if (st == DSPARK_OK) st = mark_copied(inputs_copied, s);
    if (st == DSPARK_OK) st = dspark_conf_probe(w_q8_0, hid_d, bias, threshold, K, n_probes, logit_d, gate_d, stream);
    if (st == DSPARK_OK) st = copy(gate_host, gate_d, n * 4, cudaMemcpyDeviceToHost, s, "conf_probe_host: gate copy");
    if (st == DSPARK_OK && logit_host)
        st = copy(logit_host, logit_d, n * 4, cudaMemcpyDeviceToHost, s, "conf_probe_host: logit copy");
    return st;
}

extern "C" size_t dspark_ws_matvec_host_scratch_bytes(int M, int N, int K) {
    if (M < 0 || N < 0 || K < 0) return 0;
    const size_t ws = dspark_ws_matvec_workspace_bytes(M, N, K);
    if (ws == 0) return 0;
    return up256(ws) + up256(static_cast<size_t>(M) * K * 2) + up256(static_cast<size_t>(M) * N * 4);
}

extern "C" dspark_status dspark_ws_matvec_host(const uint16_t *W, const uint16_t *X_host, void *Y_host, int y_is_fp32,
                                               int M, int N, int K, void *device_scratch, size_t scratch_bytes,
                                               void *inputs_copied, dspark_stream_t stream) {
    using namespace dspark;
    clear_error();
    if (M < 0 || N < 0 || K < 0) return fail(DSPARK_ERR_INVALID, "ws_matvec_host: negative size");
    if (M > 16) return fail(DSPARK_ERR_UNSUPPORTED, "ws_matvec_host: M=%d > 16", M);
    if (K < 8 || (K % 8) != 0) return fail(DSPARK_ERR_INVALID, "ws_matvec_host: K=%d must be a positive multiple of 8", K);
    if (M == 0 || N == 0) return DSPARK_OK;
    if (!W || !X_host || !Y_host || !device_scratch) return fail(DSPARK_ERR_INVALID, "ws_matvec_host: null pointer argument");
    if (!aligned(W, 16) || !aligned(device_scratch, 256))
        return fail(DSPARK_ERR_INVALID, "ws_matvec_host: W must be 16-byte and scratch 256-byte aligned");
    const size_t need = dspark_ws_matvec_host_scratch_bytes(M, N, K);
    if (need == 0) return fail(DSPARK_ERR_CUDA, "ws_matvec_host: could not size the scratch");
    if (scratch_bytes < need)
        return fail(DSPARK_ERR_INVALID, "ws_matvec_host: scratch of %zu bytes < required %zu", scratch_bytes, need);
    // the matvec workspace (its status word) comes first, at offset 0 for every shape that
    // shares the scratch
    const size_t ws = dspark_ws_matvec_workspace_bytes(M, N, K);
    unsigned char *p = static_cast<unsigned char *>(device_scratch);
    unsigned char *x_d = p + up256(ws);
    unsigned char *y_d = x_d + up256(static_cast<size_t>(M) * K * 2);
    const size_t ybytes = static_cast<size_t>(M) * N * (y_is_fp32 ? 4 : 2);
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    dspark_status st = copy(x_d, X_host, static_cast<size_t>(M) * K * 2, cudaMemcpyHostToDevice, s, "ws_matvec_host: X copy");
    if (st == DSPARK_OK) st = mark_copied(inputs_copied, s);
    if (st == DSPARK_OK)
        st = dspark_ws_matvec(W, reinterpret_cast<const uint16_t *>(x_d), y_d, y_is_fp32, M, N, K, p, ws, stream);
    if (st == DSPARK_OK) st = copy(Y_host, y_d, ybytes, cudaMemcpyDeviceToHost, s, "ws_matvec_host: Y copy");
    return st;
}

extern "C" size_t dspark_ws_matvec_grouped_host_scratch_bytes(const dspark_ws_problem *problems, int n_problems) {
    if (n_problems < 0 || (n_problems > 0 && !problems)) return 0;
    const size_t ws = dspark_ws_matvec_grouped_workspace_bytes(problems, n_problems);
    if (ws == 0) return 0;
    size_t bytes = up256(ws);
    for (int i = 0; i < n_problems; ++i) {
        const dspark_ws_problem &q = problems[i];
        if (q.M <= 0 || q.N <= 0 || q.K <= 0) continue;
        bytes += up256(static_cast<size_t>(q.M) * q.K * 2) + up256(static_cast<size_t>(q.M) * q.N * 4);
    }
    return bytes;
}

extern "C" dspark_status dspark_ws_matvec_grouped_host(const dspark_ws_problem *problems, int n_problems,
                                                       void *device_scratch, size_t scratch_bytes,
                                                       void *inputs_copied, dspark_stream_t stream) {
    using namespace dspark;
    clear_error();
    if (n_problems < 0 || n_problems > 8)
        return fail(DSPARK_ERR_UNSUPPORTED, "ws_matvec_grouped_host: %d problems (at most 8)", n_problems);
    if (n_problems > 0 && !problems) return fail(DSPARK_ERR_INVALID, "ws_matvec_grouped_host: null problem array");
    int live = 0;
    for (int i = 0; i < n_problems; ++i) {
        const dspark_ws_problem &q = problems[i];
        if (q.M < 0 || q.N < 0 || q.K < 0) return fail(DSPARK_ERR_INVALID, "ws_matvec_grouped_host: negative size");
        if (q.M > 16) return fail(DSPARK_ERR_UNSUPPORTED, "ws_matvec_grouped_host: M=%d > 16", q.M);
        if (q.K < 8 || (q.K % 8) != 0)
            return fail(DSPARK_ERR_INVALID, "ws_matvec_grouped_host: K=%d must be a positive multiple of 8", q.K);
        if (q.M == 0 || q.N == 0) continue;
        if (!q.W || !q.X || !q.Y) return fail(DSPARK_ERR_INVALID, "ws_matvec_grouped_host: null pointer argument");
        if (!aligned(q.W, 16)) return fail(DSPARK_ERR_INVALID, "ws_matvec_grouped_host: W must be 16-byte aligned");
        ++live;
    }
    if (live == 0) return DSPARK_OK;
    if (!device_scratch) return fail(DSPARK_ERR_INVALID, "ws_matvec_grouped_host: null scratch");
    if (!aligned(device_scratch, 256)) return fail(DSPARK_ERR_INVALID, "ws_matvec_grouped_host: scratch must be 256-byte aligned");
    const size_t need = dspark_ws_matvec_grouped_host_scratch_bytes(problems, n_problems);
    if (need == 0) return fail(DSPARK_ERR_CUDA, "ws_matvec_grouped_host: could not size the scratch");
    if (scratch_bytes < need)
        return fail(DSPARK_ERR_INVALID, "ws_matvec_grouped_host: scratch of %zu bytes < required %zu", scratch_bytes, need);
    // the grouped workspace first (its status word at offset 0), then per problem
    // the device copies of X and Y
    const size_t ws = dspark_ws_matvec_grouped_workspace_bytes(problems, n_problems);
    unsigned char *p = static_cast<unsigned char *>(device_scratch) + up256(ws);
    dspark_ws_problem dev[8];
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    dspark_status st = DSPARK_OK;
    for (int i = 0; i < n_problems; ++i) {
        dev[i] = problems[i];
        const dspark_ws_problem &q = problems[i];
        if (q.M == 0 || q.N == 0) continue;
        const size_t xb = static_cast<size_t>(q.M) * q.K * 2;
        dev[i].X = reinterpret_cast<const uint16_t *>(p);
        p += up256(xb);
        dev[i].Y = p;
        p += up256(static_cast<size_t>(q.M) * q.N * 4);
        if (st == DSPARK_OK) st = copy(const_cast<uint16_t *>(dev[i].X), q.X, xb, cudaMemcpyHostToDevice, s,
                                       "ws_matvec_grouped_host: X copy");
    }
    if (st == DSPARK_OK) st = mark_copied(inputs_copied, s);
    if (st == DSPARK_OK) st = dspark_ws_matvec_grouped(dev, n_problems, device_scratch, ws, stream);
    for (int i = 0; i < n_problems && st == DSPARK_OK; ++i) {
        const dspark_ws_problem &q = problems[i];
        if (q.M == 0 || q.N == 0) continue;
        st = copy(q.Y, dev[i].Y, static_cast<size_t>(q.M) * q.N * (q.y_is_fp32 ? 4 : 2), cudaMemcpyDeviceToHost, s,
                  "ws_matvec_grouped_host: Y copy");
    }
    return st;
}

