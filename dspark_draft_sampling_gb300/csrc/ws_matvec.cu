// Weight-stationary small-M fp16 matvec: Y[M, N] = X[M, K] . W[N, K]^T.
//
// Method (SharpInference issue #441, sections "Observation", "Hypothesis" and "Proposed
// work"): the draft's fp16 projections have M = B = 7 rows; at that M a GEMM library
// tile wastes bandwidth, so each weight element should be read from HBM once and
// applied to all M rows.
//
// GB300 design
//  * Persistent grid (at most one CTA per SM); CTA c owns the contiguous output rows
//    [c*N/G, (c+1)*N/G), processed in groups of TN rows.
//  * A producer warp streams each group's W rows through a 4-stage shared-memory ring
//    with 1-D TMA bulk copies: one stage = TN rows x 2048 k-elements (32 KB at TN = 8).
//  * Eight consumer warps split each stage's k-range (warp w: 256 elements, 8 per lane);
//    every weight element is converted to fp32 once and multiplied into all M rows with
//    packed fp32x2 FMAs (two rows of X per instruction).  X (a few tens of KB) is read
//    through L1/L2 and converted once per stage.
//  * Lane partials are combined by a fixed butterfly, warp partials by an in-order sum
//    in shared memory: each output has one summation order, independent of M, N and the
//    grid size.
#include <cuda_fp16.h>

#include "common.cuh"

namespace dspark {
namespace {

constexpr int kWarpsC = 8;
constexpr int kThreadsC = kWarpsC * 32;
constexpr int kThreads = kThreadsC + 32;
constexpr int kStages = 4;
constexpr int kKC = kWarpsC * 256;  // k-elements per stage

struct WsArgs {
    const uint16_t *W;
    const uint16_t *X;
    void *Y;
    int y_fp32;
    int M, N, K;
    unsigned *status;  // unused for now (no cross-CTA waits); kept null
    unsigned long long timeout_ns;
};

template <int TN>
constexpr size_t ws_smem_bytes(int mp) {
    return size_t(kStages) * TN * kKC * 2 + size_t(kWarpsC) * TN * mp * sizeof(float) +
           2 * kStages * sizeof(uint64_t) + 16;
}

__device__ __forceinline__ float2 h2f(uint32_t w) {
    __half2 h = *reinterpret_cast<__half2 *>(&w);
    return __half22float2(h);
}

template <int MP, int TN>
__global__ void __launch_bounds__(kThreads, 1) ws_matvec_kernel(WsArgs a) {
    constexpr int SB = TN * kKC * 2;  // stage bytes
    constexpr int NV = TN * MP;       // partial sums per lane
    extern __shared__ __align__(128) unsigned char smem[];
    unsigned char *ring = smem;
    float *red = reinterpret_cast<float *>(smem + size_t(kStages) * SB);  // [kWarpsC][NV]
    uint64_t *full = reinterpret_cast<uint64_t *>(red + kWarpsC * NV);
    uint64_t *empty = full + kStages;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int nctas = gridDim.x;
    const int cta = blockIdx.x;
    const int n0 = static_cast<int>(static_cast<long long>(cta) * a.N / nctas);
    const int n1 = static_cast<int>(static_cast<long long>(cta + 1) * a.N / nctas);
    const int rows_c = n1 - n0;
    const int ngroups = (rows_c + TN - 1) / TN;
    const int nkc = (a.K + kKC - 1) / kKC;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], kWarpsC);
        }
        fence_mbar_init();
    }
    __syncthreads();

    if (warp == kWarpsC) {  // producer
        if (lane == 0) {
            const uint64_t pol = l2_policy_evict_first();
            int stage = 0;
            uint32_t phase = 0;
            for (int g = 0; g < ngroups; ++g) {
                const int vrows = min(TN, rows_c - g * TN);
                for (int kc = 0; kc < nkc; ++kc) {
                    if (!mbar_wait(&empty[stage], phase ^ 1u, a.timeout_ns)) return;
                    const int klen = min(kKC, a.K - kc * kKC);
                    const uint32_t row_bytes = static_cast<uint32_t>(klen) * 2u;
                    mbar_arrive_expect_tx(&full[stage], row_bytes * vrows);
                    for (int t = 0; t < vrows; ++t)
                        bulk_g2s(ring + size_t(stage) * SB + size_t(t) * kKC * 2,
                                 a.W + size_t(n0 + g * TN + t) * a.K + size_t(kc) * kKC, row_bytes, &full[stage],
                                 pol);
                    if (++stage == kStages) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
        }
        return;
    }

    int stage = 0;
    uint32_t phase = 0;
    bool broken = false;  // a tile wait timed out: wait on no further tiles (results undefined)
    const int M = a.M;
    for (int g = 0; g < ngroups; ++g) {
        const int vrows = min(TN, rows_c - g * TN);
        float2 acc[TN][MP / 2];
#pragma unroll
        for (int t = 0; t < TN; ++t)
#pragma unroll
            for (int mp = 0; mp < MP / 2; ++mp) acc[t][mp] = make_float2(0.f, 0.f);

        for (int kc = 0; kc < nkc; ++kc) {
            const int kl = warp * 256 + lane * 8;  // this lane's k offset inside the stage
            const int k0 = kc * kKC + kl;
            const bool active = k0 < a.K;
            uint32_t xh[MP][4];
#pragma unroll
            for (int m = 0; m < MP; ++m) {
                uint4 u = make_uint4(0u, 0u, 0u, 0u);
                if (active && m < M) u = *reinterpret_cast<const uint4 *>(a.X + size_t(m) * a.K + k0);
                xh[m][0] = u.x;
                xh[m][1] = u.y;
                xh[m][2] = u.z;
                xh[m][3] = u.w;
            }
            if (!broken && !mbar_wait(&full[stage], phase, a.timeout_ns)) broken = true;
            if (active && !broken) {
                const unsigned char *st = ring + size_t(stage) * SB;
                uint32_t wh[TN][4];
#pragma unroll
                for (int t = 0; t < TN; ++t) {
                    uint4 u = make_uint4(0u, 0u, 0u, 0u);
                    if (t < vrows) u = *reinterpret_cast<const uint4 *>(st + size_t(t) * kKC * 2 + size_t(kl) * 2);
                    wh[t][0] = u.x;
                    wh[t][1] = u.y;
                    wh[t][2] = u.z;
                    wh[t][3] = u.w;
                }
#pragma unroll
                for (int e2 = 0; e2 < 4; ++e2) {
                    float2 xe[MP / 2], xo[MP / 2];
#pragma unroll
                    for (int mp = 0; mp < MP / 2; ++mp) {
                        const float2 f0 = h2f(xh[2 * mp][e2]);
                        const float2 f1 = h2f(xh[2 * mp + 1][e2]);
                        xe[mp] = make_float2(f0.x, f1.x);
                        xo[mp] = make_float2(f0.y, f1.y);
                    }
#pragma unroll
                    for (int t = 0; t < TN; ++t) {
                        if (t < vrows) {
                            const float2 wf = h2f(wh[t][e2]);
                            const float2 wa = make_float2(wf.x, wf.x);
                            const float2 wb = make_float2(wf.y, wf.y);
#pragma unroll
                            for (int mp = 0; mp < MP / 2; ++mp) {
                                acc[t][mp] = __ffma2_rn(wa, xe[mp], acc[t][mp]);
                                acc[t][mp] = __ffma2_rn(wb, xo[mp], acc[t][mp]);
                            }
                        }
                    }
                }
            }
            __syncwarp();
            if (lane == 0 && !broken) mbar_arrive(&empty[stage]);
            if (++stage == kStages) {
                stage = 0;
                phase ^= 1u;
            }
        }

        float vals[NV];
#pragma unroll
        for (int t = 0; t < TN; ++t)
#pragma unroll
            for (int mp = 0; mp < MP / 2; ++mp) {
                vals[t * MP + 2 * mp] = acc[t][mp].x;
                vals[t * MP + 2 * mp + 1] = acc[t][mp].y;
            }
        ReduceScatter<NV, 16>::run(vals, lane);
        constexpr int LEFT = rs_values_left<NV, 16>();
        const int first = rs_first_index<NV, 16>(lane);
#pragma unroll
        for (int j = 0; j < LEFT; ++j) red[warp * NV + first + j] = vals[j];
        named_bar_sync(1, kThreadsC);
        for (int idx = threadIdx.x; idx < NV; idx += kThreadsC) {
            const int t = idx / MP;
            const int m = idx % MP;
            if (t < vrows && m < M) {
                float s = red[idx];
#pragma unroll
                for (int w = 1; w < kWarpsC; ++w) s += red[w * NV + idx];
                const size_t o = size_t(m) * a.N + (n0 + g * TN + t);
                if (a.y_fp32)
                    static_cast<float *>(a.Y)[o] = s;
                else
                    static_cast<__half *>(a.Y)[o] = __float2half_rn(s);
            }
        }
        named_bar_sync(1, kThreadsC);
    }
}

template <int MP, int TN>
dspark_status launch_ws(const WsArgs &args, int nctas, cudaStream_t stream) {
    auto kern = ws_matvec_kernel<MP, TN>;
    const size_t smem = ws_smem_bytes<TN>(MP);
    static int configured_dev = -1;
    int dev = 0;
    cudaGetDevice(&dev);
    if (configured_dev != dev) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
        if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute(ws_matvec)");
        configured_dev = dev;
    }
    kern<<<nctas, kThreads, smem, stream>>>(args);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(e, "ws_matvec launch");
    return DSPARK_OK;
}

}  // namespace
}  // namespace dspark

extern "C" dspark_status dspark_ws_matvec(const uint16_t *W, const uint16_t *X, void *Y, int y_is_fp32, int M, int N,
                                          int K, dspark_stream_t stream) {
    using namespace dspark;
    clear_error();
    if (M < 0 || N < 0 || K < 0) return fail(DSPARK_ERR_INVALID, "ws_matvec: negative size");
    if (M > 16) return fail(DSPARK_ERR_UNSUPPORTED, "ws_matvec: M=%d > 16", M);
    if (K < 8 || (K % 8) != 0) return fail(DSPARK_ERR_INVALID, "ws_matvec: K=%d must be a positive multiple of 8", K);
    if (M == 0 || N == 0) return DSPARK_OK;  // nothing to enqueue
    if (!W || !X || !Y) return fail(DSPARK_ERR_INVALID, "ws_matvec: null pointer argument");
    if (!aligned(W, 16) || !aligned(X, 16)) return fail(DSPARK_ERR_INVALID, "ws_matvec: W and X must be 16-byte aligned");
    if (!aligned(Y, y_is_fp32 ? 4 : 2)) return fail(DSPARK_ERR_INVALID, "ws_matvec: misaligned Y");
    int sms = 0;
    int rc = current_sm_count(&sms);
    if (rc != DSPARK_OK) return static_cast<dspark_status>(rc);
    WsArgs args;
    args.W = W;
    args.X = X;
    args.Y = Y;
    args.y_fp32 = y_is_fp32 ? 1 : 0;
    args.M = M;
    args.N = N;
    args.K = K;
    args.status = nullptr;
    args.timeout_ns = kDefaultTimeoutNs;
    const int nctas = N < sms ? N : sms;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (M <= 2) return launch_ws<2, 8>(args, nctas, s);
    if (M <= 4) return launch_ws<4, 8>(args, nctas, s);
    if (M <= 8) return launch_ws<8, 8>(args, nctas, s);
    return launch_ws<16, 4>(args, nctas, s);
}
