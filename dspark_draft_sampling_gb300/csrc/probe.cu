// Proposer confidence probe: Q8_0 dequant-dot of the hidden state + logit-space gate.
//
// Method (ds4 PR #772 "dspark: cut per-cycle CUDA overheads", sections "Summary" and
// "Root cause"): a 7424-wide matvec of the hidden vector against Q8_0 weights, run on
// the GPU so that only a 4-byte gate decision crosses to the host.
//
// One CTA of 256 threads per probe.  Thread t walks the 16-byte chunks t, t + 256, ... of the
// hidden vector (one vector load each), dequantizes the matching four int8 weights with their
// block's fp16 scale exactly in fp32, and accumulates in chunk order; a fixed warp butterfly
// plus an in-order sum of the eight warp totals gives z.  Two load schedules, the same
// arithmetic in the same order (so the same bits): for a large batch a loop unrolled four
// times (many CTAs resident, few registers each), for a small batch or a single probe every
// chunk load of a thread issued before any is used (one memory latency per probe).  The gate
// compares z with logit(threshold) (computed on the host), which is the same decision as
// sigmoid(z) >= threshold without evaluating an exponential on the device.
#include <cuda_fp16.h>

#include <cmath>

#include "common.cuh"

namespace dspark {
namespace {

constexpr int kProbeThreads = 256;
constexpr int kProbeWarps = kProbeThreads / 32;
constexpr int kAhead = 8;  // small batches: chunk loads per thread in flight together

__device__ __forceinline__ float4 ldg_stream_f4(const float *p) {
    const uint4 u = ldg_nc_v4(p);
    return make_float4(__uint_as_float(u.x), __uint_as_float(u.y), __uint_as_float(u.z), __uint_as_float(u.w));
}

// acc += d * (q0 x0 + q1 x1 + q2 x2 + q3 x3) for chunk c, the weights read from its Q8_0 block
__device__ __forceinline__ float probe_chunk(const uint8_t *__restrict__ wq, int c, float4 xv, float acc) {
    const uint8_t *blk = wq + size_t(c >> 3) * 34;
    const int off = 2 + 4 * (c & 7);
    const unsigned short dbits = static_cast<unsigned short>(__ldg(blk) | (__ldg(blk + 1) << 8));
    const float d = __half2float(__ushort_as_half(dbits));
    const float q0 = static_cast<float>(static_cast<int8_t>(__ldg(blk + off + 0)));
    const float q1 = static_cast<float>(static_cast<int8_t>(__ldg(blk + off + 1)));
    const float q2 = static_cast<float>(static_cast<int8_t>(__ldg(blk + off + 2)));
    const float q3 = static_cast<float>(static_cast<int8_t>(__ldg(blk + off + 3)));
    float s = q0 * xv.x;
    s = fmaf(q1, xv.y, s);
    s = fmaf(q2, xv.z, s);
    s = fmaf(q3, xv.w, s);
    return fmaf(d, s, acc);
}

// The probe's input vector may come in two pieces (the hidden state and the Markov
// state): chunk c < nchunks_a reads piece a, the rest read piece b.  With one piece
// (nchunks_b == 0) this is the plain contiguous probe; the chunk order, and so every
// rounding, is the same either way.
template <bool kAllAhead>
__global__ void __launch_bounds__(kProbeThreads)
    conf_probe_kernel(const uint8_t *__restrict__ wq, const float *__restrict__ xa, long long lda, int nchunks_a,
                      const float *__restrict__ xb, long long ldb, int nchunks_b, float bias, float t_logit,
                      float *logit_out, int32_t *gate_out, cudaGraphConditionalHandle cond, int set_cond) {
    pdl_launch_dependents();
    pdl_wait();
    __shared__ float warp_sum[kProbeWarps];
    const float *pa = xa + size_t(blockIdx.x) * lda;
    const float *pb = xb ? xb + size_t(blockIdx.x) * ldb : nullptr;
    const int nchunks = nchunks_a + nchunks_b;  // 4 floats per chunk; a Q8_0 block spans 8 chunks
    auto chunk_ptr = [&](int c) { return c < nchunks_a ? pa + 4 * c : pb + 4 * (c - nchunks_a); };
    float acc = 0.f;
    if constexpr (kAllAhead) {
        for (int c0 = threadIdx.x; c0 < nchunks; c0 += kAhead * kProbeThreads) {
            float4 xv[kAhead];
#pragma unroll
            for (int u = 0; u < kAhead; ++u) {
                const int c = c0 + u * kProbeThreads;
                xv[u] = c < nchunks ? ldg_stream_f4(chunk_ptr(c)) : make_float4(0.f, 0.f, 0.f, 0.f);
            }
#pragma unroll
            for (int u = 0; u < kAhead; ++u) {
                const int c = c0 + u * kProbeThreads;
                if (c < nchunks) acc = probe_chunk(wq, c, xv[u], acc);
            }
        }
    } else {
#pragma unroll 4
        for (int c = threadIdx.x; c < nchunks; c += kProbeThreads) acc = probe_chunk(wq, c, ldg_stream_f4(chunk_ptr(c)), acc);
    }
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
    if ((threadIdx.x & 31) == 0) warp_sum[threadIdx.x >> 5] = acc;
    __syncthreads();
    if (threadIdx.x == 0) {
        float z = warp_sum[0];
#pragma unroll
        for (int w = 1; w < kProbeWarps; ++w) z += warp_sum[w];
        z += bias;
        const int gate = (z >= t_logit) ? 1 : 0;
        if (logit_out) logit_out[blockIdx.x] = z;
        gate_out[blockIdx.x] = gate;
        // inside a gated draft graph: probe 0's decision selects whether the draft runs
        if (set_cond && blockIdx.x == 0) cudaGraphSetConditional(cond, static_cast<unsigned>(gate));
    }
}

}  // namespace

dspark_status probe_enqueue(const void *w_q8_0, const float *xa, int Ka, long long lda, const float *xb, int Kb,
                            long long ldb, float bias, float threshold, int n_probes, float *logit_out,
                            int32_t *gate_out, cudaStream_t stream, cudaGraphConditionalHandle cond,
                            int set_cond) {
    clear_error();
    const int K = Ka + Kb;
    if (Ka <= 0 || Kb < 0 || (K % 32) != 0 || (Ka % 4) != 0 || (Kb % 4) != 0)
        return fail(DSPARK_ERR_INVALID, "conf_probe: widths %d + %d must be multiples of 4 summing to a multiple of 32",
                    Ka, Kb);
    if (n_probes < 0) return fail(DSPARK_ERR_INVALID, "conf_probe: n_probes=%d < 0", n_probes);
    if (!(threshold > 0.f && threshold < 1.f))
        return fail(DSPARK_ERR_INVALID, "conf_probe: threshold must lie in (0, 1)");
    if (n_probes == 0) return DSPARK_OK;  // nothing to enqueue
    if (!w_q8_0 || !xa || (Kb > 0 && !xb) || !gate_out)
        return fail(DSPARK_ERR_INVALID, "conf_probe: null pointer argument");
    if (!aligned(xa, 16) || (Kb > 0 && !aligned(xb, 16)) || (lda % 4) != 0 || (Kb > 0 && (ldb % 4) != 0) ||
        lda < Ka || (Kb > 0 && ldb < Kb))
        return fail(DSPARK_ERR_INVALID, "conf_probe: inputs must be 16-byte aligned with row strides >= widths");
    if (!aligned(gate_out, 4) || (logit_out && !aligned(logit_out, 4)))
        return fail(DSPARK_ERR_INVALID, "conf_probe: misaligned output pointer");
    // logit(t) on the host in double: sigmoid(z) >= t  <=>  z >= log(t / (1 - t)).
    const double t = static_cast<double>(threshold);
    const float t_logit = static_cast<float>(std::log(t / (1.0 - t)));
    const uint8_t *wb = static_cast<const uint8_t *>(w_q8_0);
    const float *xbp = Kb > 0 ? xb : nullptr;
    // all loads of a thread in flight together while the batch fits in one wave of CTAs
    int sms = 0;
    int rc = current_sm_count(&sms);
    if (rc != DSPARK_OK) return static_cast<dspark_status>(rc);
    const bool ahead = n_probes <= 8 * sms;
    auto kern = ahead ? conf_probe_kernel<true> : conf_probe_kernel<false>;
    cudaError_t e;
    if (set_cond) {  // inside a conditional graph: plain launch
        kern<<<n_probes, kProbeThreads, 0, stream>>>(wb, xa, lda, Ka / 4, xbp, ldb, Kb / 4, bias, t_logit, logit_out,
                                                     gate_out, cond, set_cond);
        e = cudaGetLastError();
    } else {
        e = launch_pdl(kern, dim3(static_cast<unsigned>(n_probes)), dim3(kProbeThreads), 0, stream, wb, xa, lda,
                       Ka / 4, xbp, ldb, Kb / 4, bias, t_logit, logit_out, gate_out, cond, set_cond);
    }
    if (e != cudaSuccess) return cuda_fail(e, "conf_probe launch");
    return DSPARK_OK;
}

}  // namespace dspark

extern "C" dspark_status dspark_conf_probe(const void *w_q8_0, const float *hidden, float bias, float threshold,
                                           int K, int n_probes, float *logit_out, int32_t *gate_out,
                                           dspark_stream_t stream) {
    if (K <= 0 || (K % 32) != 0) {
        dspark::clear_error();
        return dspark::fail(DSPARK_ERR_INVALID, "conf_probe: K=%d must be a positive multiple of 32", K);
    }
    return dspark::probe_enqueue(w_q8_0, hidden, K, K, nullptr, 0, 0, bias, threshold, n_probes, logit_out, gate_out,
                                 reinterpret_cast<cudaStream_t>(stream), 0ull, 0);
}

extern "C" dspark_status dspark_conf_probe_split(const void *w_q8_0, const float *hidden, int K_hidden,
                                                 long long ld_hidden, const float *state, int K_state,
                                                 long long ld_state, float bias, float threshold, int n_probes,
                                                 float *logit_out, int32_t *gate_out, dspark_stream_t stream) {
    return dspark::probe_enqueue(w_q8_0, hidden, K_hidden, ld_hidden, state, K_state, ld_state, bias, threshold,
                                 n_probes, logit_out, gate_out, reinterpret_cast<cudaStream_t>(stream), 0ull, 0);
}
