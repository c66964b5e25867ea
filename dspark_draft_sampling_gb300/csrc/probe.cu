// Proposer confidence probe: Q8_0 dequant-dot of the hidden state + logit-space gate.
//
// Method (ds4 PR #772 "dspark: cut per-cycle CUDA overheads", sections "Summary" and
// "Root cause"): a 7424-wide matvec of the hidden vector against Q8_0 weights, run on
// the GPU so that only a 4-byte gate decision crosses to the host.
//
// One CTA of 256 threads per probe.  Thread t walks the 16-byte chunks t, t + 256, ... of the
// hidden vector (one vector load each), dequantizes the matching four int8 weights with their
// block's fp16 scale exactly in fp32, and accumulates in chunk order; a fixed warp butterfly
// plus an in-order sum of the eight warp totals gives z.  Three load schedules, the same
// arithmetic in the same order (so the same bits): for a small batch or a single probe every
// chunk load of a thread issued before any is used (one memory latency per probe); for a
// large batch persistent CTAs (one per SM) that stage the Q8_0 row in shared memory by a bulk
// copy, decode it once, and stream whole hidden rows through a ring of bulk copies
// (cp.async.bulk, one thread issuing, several rows in flight per SM) to two groups of 256
// threads taking alternate probes; or, when the ring does not fit shared memory, a loop
// unrolled four times with one CTA per probe.  The gate
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

// ---- large batches: persistent CTAs, hidden rows through a ring of bulk copies ----------
// Two consumer groups of 256 threads take alternate probes (each group does the arithmetic of
// conf_probe_kernel for its probe); warp 16 issues the copies.
constexpr int kRingGroups = 2;
constexpr int kRingConsumers = kRingGroups * kProbeThreads;
constexpr int kRingThreads = kRingConsumers + 32;
constexpr int kRingMaxSlots = 8;
constexpr size_t kRingSmemBudget = 227 * 1024;

__device__ __forceinline__ void bulk_copy_g2s(void *dst, const void *src, uint32_t bytes, uint64_t *bar) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                     smem_addr(dst)),
                 "l"(src), "r"(bytes), "r"(smem_addr(bar))
                 : "memory");
}

// Block scales padded to 16 bytes, so the ring (bulk-copy destinations) stays 16-byte aligned.
__host__ __device__ inline size_t ring_scale_bytes(int nchunks) { return (size_t(nchunks / 8) * 4 + 15) / 16 * 16; }
// The raw Q8_0 row staged for decoding: its bytes plus up to 15 on either side of the
// 16-byte-aligned interior that the bulk copy moves.
__host__ __device__ inline size_t ring_raw_bytes(int nchunks) { return (size_t(nchunks / 8) * 34 + 32 + 15) / 16 * 16; }

// Shared memory: the decoded weights (q as 4 floats per chunk, d per block), the ring of
// nslots hidden rows, the raw Q8_0 row, the barriers and the warp totals.
size_t ring_smem_bytes(int nchunks, int nslots) {
    return 128 + size_t(nchunks) * 16 + ring_scale_bytes(nchunks) + size_t(nslots) * nchunks * 16 +
           ring_raw_bytes(nchunks) + (2 * kRingMaxSlots + 1) * 8 + kRingGroups * 2 * kProbeWarps * 4 + 16;
}

__global__ void __launch_bounds__(kRingThreads, 1)
    conf_probe_ring_kernel(const uint8_t *__restrict__ wq, const float *__restrict__ xa, long long lda, int nchunks_a,
                           const float *__restrict__ xb, long long ldb, int nchunks_b, float bias, float t_logit,
                           float *logit_out, int32_t *gate_out, int n_probes, int nslots,
                           unsigned long long timeout_ns) {
    extern __shared__ unsigned char smem_raw[];
    unsigned char *sm = smem_raw + ((128u - (smem_addr(smem_raw) & 127u)) & 127u);
    const int nchunks = nchunks_a + nchunks_b;
    const int nbytes = (nchunks / 8) * 34;                               // the Q8_0 row
    float4 *wq4 = reinterpret_cast<float4 *>(sm);                        // [nchunks] q as floats
    float *wd = reinterpret_cast<float *>(wq4 + nchunks);                // [nchunks / 8] block scales
    float4 *ring = reinterpret_cast<float4 *>(reinterpret_cast<unsigned char *>(wd) +
                                              ring_scale_bytes(nchunks));  // [nslots][nchunks] hidden rows
    unsigned char *raw = reinterpret_cast<unsigned char *>(ring + size_t(nslots) * nchunks);
    uint64_t *full = reinterpret_cast<uint64_t *>(raw + ring_raw_bytes(nchunks));
    uint64_t *empty = full + kRingMaxSlots;
    uint64_t *wbar = empty + kRingMaxSlots;                              // the raw row landed
    float *warp_sum = reinterpret_cast<float *>(wbar + 1);               // [groups][2][kProbeWarps]
    int *s_abort = reinterpret_cast<int *>(warp_sum + kRingGroups * 2 * kProbeWarps);
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    // the row's 16-byte-aligned interior [ia, ib) goes by bulk copy, to raw + (ia - row0) where
    // row0 = wq - lead keeps that destination 16-byte aligned; the ragged ends by byte loads
    const uintptr_t w0 = reinterpret_cast<uintptr_t>(wq);
    const uintptr_t ia = (w0 + 15) & ~uintptr_t(15);
    const uintptr_t ib = (w0 + nbytes) & ~uintptr_t(15);
    const int lead = static_cast<int>(w0 & 15);  // raw[lead + i] holds row byte i
    const bool interior = ib > ia;

    if (threadIdx.x == kRingConsumers) {
        for (int q = 0; q < kRingMaxSlots; ++q) {
            mbar_init(&full[q], 1);
            mbar_init(&empty[q], 1);
        }
        mbar_init(wbar, 1);
        *s_abort = 0;
        fence_mbar_init();
    }
    __syncthreads();
    pdl_launch_dependents();
    pdl_wait();  // no global-memory access before this point

    if (warp == kRingConsumers / 32) {
        // ---- copy issuer: the weight row, then the CTA's probes p = blockIdx.x, + gridDim.x, ... ----
        if (lane == 0) {
            if (interior) {
                mbar_arrive_expect_tx(wbar, static_cast<uint32_t>(ib - ia));
                bulk_copy_g2s(raw + lead + (ia - w0), reinterpret_cast<const void *>(ia), static_cast<uint32_t>(ib - ia),
                              wbar);
            }
            const uint32_t bytes = static_cast<uint32_t>(nchunks) * 16u;
            int j = 0;
            for (int p = blockIdx.x; p < n_probes; p += gridDim.x, ++j) {
                const int q = j % nslots;
                if (j >= nslots && !mbar_wait(&empty[q], static_cast<uint32_t>((j / nslots) & 1) ^ 1u, timeout_ns)) {
                    *reinterpret_cast<volatile int *>(s_abort) = 1;
                    break;
                }
                if (*reinterpret_cast<volatile int *>(s_abort)) break;
                float4 *dst = ring + size_t(q) * nchunks;
                mbar_arrive_expect_tx(&full[q], bytes);
                bulk_copy_g2s(dst, xa + size_t(p) * lda, static_cast<uint32_t>(nchunks_a) * 16u, &full[q]);
                if (nchunks_b)
                    bulk_copy_g2s(dst + nchunks_a, xb + size_t(p) * ldb, static_cast<uint32_t>(nchunks_b) * 16u,
                                  &full[q]);
            }
            // copies still in flight land before the CTA exits
            for (int i = j > nslots ? j - nslots : 0; i < j; ++i)
                mbar_wait(&full[i % nslots], static_cast<uint32_t>((i / nslots) & 1), timeout_ns);
            if (interior) mbar_wait(wbar, 0, timeout_ns);
        }
        return;
    }
    // ---- consumers: decode the Q8_0 row once (from shared memory), then one probe per slot ----
    const int t = threadIdx.x;  // 0 .. kRingConsumers - 1
    {
        // ragged ends of the row (at most 15 bytes each) by byte loads
        const int head = interior ? static_cast<int>(ia - w0) : nbytes;
        const int tail0 = interior ? static_cast<int>(ib - w0) : nbytes;
        for (int i = t; i < head; i += kRingConsumers) raw[lead + i] = __ldg(wq + i);
        for (int i = tail0 + t; i < nbytes; i += kRingConsumers) raw[lead + i] = __ldg(wq + i);
        bool ok = !interior || mbar_wait(wbar, 0, timeout_ns);
        if (!ok) *reinterpret_cast<volatile int *>(s_abort) = 1;
        named_bar_sync(3, kRingConsumers);
        const unsigned char *rw = raw + lead;
        for (int c = t; c < nchunks; c += kRingConsumers) {
            const unsigned char *blk = rw + size_t(c >> 3) * 34;
            const int off = 2 + 4 * (c & 7);
            if ((c & 7) == 0) {
                const unsigned short dbits = static_cast<unsigned short>(blk[0] | (blk[1] << 8));
                wd[c >> 3] = __half2float(__ushort_as_half(dbits));
            }
            wq4[c] = make_float4(static_cast<float>(static_cast<int8_t>(blk[off + 0])),
                                 static_cast<float>(static_cast<int8_t>(blk[off + 1])),
                                 static_cast<float>(static_cast<int8_t>(blk[off + 2])),
                                 static_cast<float>(static_cast<int8_t>(blk[off + 3])));
        }
        named_bar_sync(3, kRingConsumers);
    }
    const int grp = t / kProbeThreads;
    const int tid = t - grp * kProbeThreads;  // the thread index of conf_probe_kernel
    const int gwarp = tid >> 5;
    int j = grp;
    for (int p = blockIdx.x + grp * gridDim.x; p < n_probes; p += kRingGroups * gridDim.x, j += kRingGroups) {
        const int q = j % nslots;
        bool ok = !*reinterpret_cast<volatile int *>(s_abort) &&
                  mbar_wait(&full[q], static_cast<uint32_t>((j / nslots) & 1), timeout_ns);
        float acc = 0.f;
        if (ok) {
            const float4 *x = ring + size_t(q) * nchunks;
#pragma unroll 4
            for (int c = tid; c < nchunks; c += kProbeThreads) {  // the order of conf_probe_kernel
                const float4 xv = x[c];
                const float4 w = wq4[c];
                float s = w.x * xv.x;
                s = fmaf(w.y, xv.y, s);
                s = fmaf(w.z, xv.z, s);
                s = fmaf(w.w, xv.w, s);
                acc = fmaf(wd[c >> 3], s, acc);
            }
        } else {
            *reinterpret_cast<volatile int *>(s_abort) = 1;
        }
#pragma unroll
        for (int o = 16; o >= 1; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
        float *ws = warp_sum + (grp * 2 + ((j / kRingGroups) & 1)) * kProbeWarps;
        if (lane == 0) ws[gwarp] = acc;
        named_bar_sync(1 + grp, kProbeThreads);  // the group is done with slot q and wrote its totals
        if (tid == 0) {
            mbar_arrive(&empty[q]);
            float z = ws[0];
#pragma unroll
            for (int w = 1; w < kProbeWarps; ++w) z += ws[w];
            z += bias;
            // a wait that gave up (never in normal operation): gate -1, logit NaN
            const bool good = !*reinterpret_cast<volatile int *>(s_abort);
            if (logit_out) logit_out[p] = good ? z : __int_as_float(0x7fc00000);
            gate_out[p] = good ? ((z >= t_logit) ? 1 : 0) : -1;
        }
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
    const int nchunks = K / 4;
    int nslots = 0;
    while (nslots < kRingMaxSlots && ring_smem_bytes(nchunks, nslots + 1) <= kRingSmemBudget) ++nslots;
    if (!ahead && !set_cond && nslots >= 3) {
        static int configured_dev = -1;
        int dev = 0;
        cudaError_t e = cudaGetDevice(&dev);
        if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
        if (configured_dev != dev) {
            e = cudaFuncSetAttribute(conf_probe_ring_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     static_cast<int>(kRingSmemBudget));
            if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute(conf_probe_ring)");
            configured_dev = dev;
        }
        const unsigned grid = static_cast<unsigned>(n_probes < sms ? n_probes : sms);
        e = launch_pdl(conf_probe_ring_kernel, dim3(grid), dim3(kRingThreads), ring_smem_bytes(nchunks, nslots), stream,
                       wb, xa, lda, Ka / 4, xbp, ldb, Kb / 4, bias, t_logit, logit_out, gate_out, n_probes, nslots,
                       kDefaultTimeoutNs);
        if (e != cudaSuccess) return cuda_fail(e, "conf_probe launch");
        return DSPARK_OK;
    }
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
