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
//  * Each group's W rows stream through a 6-stage shared-memory ring with 1-D TMA bulk
//    copies (one stage = TN rows x 2048 k-elements, 32 KB at TN = 8), issued by lane 0 of
//    warp 0 between its own tiles.
//  * Eight warps split each stage's k-range (warp w: 256 elements, 8 per lane);
//    every weight pair is converted to fp32 once and multiplied into all M rows with
//    packed fp32x2 FMAs over (even k, odd k) pairs, so operands are used as loaded.  X (a
//    few tens of KB) is read through L1/L2 and converted once per stage and row group.
//  * Lane partials are combined by a fixed butterfly, warp partials by an in-order sum
//    in shared memory: each output has one summation order, independent of M, N and the
//    grid size.
#include <cuda/std/type_traits>
#include <cuda_fp16.h>

#include "common.cuh"

namespace dspark {
namespace {

// 8 warps = 2 per SM sub-partition, so a thread may hold up to 255 registers.  All 8 warps
// compute; lane 0 of warp 0 also issues the TMA copies (no dedicated producer warp, which
// would put a third warp on one sub-partition and cap registers at 168).
constexpr int kWarpsC = 8;
constexpr int kThreadsC = kWarpsC * 32;
constexpr int kThreads = kThreadsC;
constexpr int kStages = 6;
constexpr int kKC = kWarpsC * 256;  // k-elements per stage

struct WsArgs {
    const uint16_t *W;
    const uint16_t *X;
    void *Y;
    int y_fp32;
    int M, N, K;
    unsigned long long timeout_ns;
};

template <int TN>
constexpr size_t ws_smem_bytes(int mt) {
    return size_t(kStages) * TN * kKC * 2 + size_t(kWarpsC) * 64 * sizeof(float) * ((TN * mt + 63) / 64) +
           2 * kStages * sizeof(uint64_t) + 16;
}

__device__ __forceinline__ float2 h2f(uint32_t w) {
    __half2 h = *reinterpret_cast<__half2 *>(&w);
    return __half22float2(h);
}

__device__ __forceinline__ bool mbar_test_wait(uint64_t *bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_addr(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

constexpr int pow2_at_least(int n) {
    int p = 1;
    while (p < n) p *= 2;
    return p;
}

template <int MT, int TN>
__global__ void __launch_bounds__(kThreads, 1) ws_matvec_kernel(WsArgs a) {
    constexpr int SB = TN * kKC * 2;        // stage bytes
    constexpr int NV = TN * MT;             // partial sums per lane
    constexpr int NVP = pow2_at_least(NV);  // padded for the butterfly
    extern __shared__ __align__(128) unsigned char smem[];
    unsigned char *ring = smem;
    float *red = reinterpret_cast<float *>(smem + size_t(kStages) * SB);  // [kWarpsC][NVP]
    uint64_t *full = reinterpret_cast<uint64_t *>(red + kWarpsC * NVP);
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
    const int ntiles = ngroups * nkc;  // tile j = (group j / nkc, k-chunk j % nkc)

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], kWarpsC);
        }
        fence_mbar_init();
    }
    __syncthreads();

    // ---- producer duty of thread 0: tile j goes to stage j % kStages once tile
    // j - kStages has been released by all warps (phase (j / kStages) - 1 of empty).
    const bool producer = threadIdx.x == 0;
    uint64_t pol = 0;
    if (producer) pol = l2_policy_evict_first();
    int issued = 0;
    bool broken = false;  // a wait timed out: stop waiting (results undefined, nothing hangs)
    auto issue = [&](int j) {
        const int g = j / nkc, kc = j % nkc, st = j % kStages;
        const int vrows = min(TN, rows_c - g * TN);
        const int klen = min(kKC, a.K - kc * kKC);
        const uint32_t row_bytes = static_cast<uint32_t>(klen) * 2u;
        mbar_arrive_expect_tx(&full[st], row_bytes * vrows);
        for (int t = 0; t < vrows; ++t)
            bulk_g2s(ring + size_t(st) * SB + size_t(t) * kKC * 2,
                     a.W + size_t(n0 + g * TN + t) * a.K + size_t(kc) * kKC, row_bytes, &full[st], pol);
    };
    auto refill = [&](int j) {  // thread 0: make sure tile j is issued, then top up the ring
        while (!broken && issued <= j) {
            if (!mbar_wait(&empty[issued % kStages], ((issued / kStages) & 1) ^ 1, a.timeout_ns)) {
                broken = true;
                break;
            }
            issue(issued++);
        }
        while (!broken && issued < ntiles && issued < j + kStages &&
               mbar_test_wait(&empty[issued % kStages], ((issued / kStages) & 1) ^ 1))
            issue(issued++);
    };

    const int M = a.M;
    const int kl = warp * 256 + lane * 8;  // this lane's k offset inside a stage

    // One stage: this lane's 8 k-elements of TN weight rows against MT rows of X.
    // acc[t][m] holds (sum over even k, sum over odd k): one fp32x2 FMA consumes a
    // weight pair and an activation pair exactly as they sit in memory.
    auto stage_fma = [&](auto full_tag, const unsigned char *st, int vrows, const uint32_t (&xh)[MT][4],
                         float2 (&acc)[TN][MT]) {
        constexpr bool FULL = decltype(full_tag)::value;
        uint32_t wh[TN][4];
#pragma unroll
        for (int t = 0; t < TN; ++t) {
            uint4 u = make_uint4(0u, 0u, 0u, 0u);
            if (FULL || t < vrows) u = *reinterpret_cast<const uint4 *>(st + size_t(t) * kKC * 2 + size_t(kl) * 2);
            wh[t][0] = u.x;
            wh[t][1] = u.y;
            wh[t][2] = u.z;
            wh[t][3] = u.w;
        }
#pragma unroll
        for (int e2 = 0; e2 < 4; ++e2) {
            float2 xp[MT];
#pragma unroll
            for (int m = 0; m < MT; ++m) xp[m] = h2f(xh[m][e2]);
#pragma unroll
            for (int t = 0; t < TN; ++t) {
                if (FULL || t < vrows) {
                    const float2 wp = h2f(wh[t][e2]);
#pragma unroll
                    for (int m = 0; m < MT; ++m) acc[t][m] = __ffma2_rn(wp, xp[m], acc[t][m]);
                }
            }
        }
    };

    int j = 0;  // tile index
    bool wbroken = false;  // this warp stopped waiting on tiles
    for (int g = 0; g < ngroups; ++g) {
        const int vrows = min(TN, rows_c - g * TN);
        float2 acc[TN][MT];
#pragma unroll
        for (int t = 0; t < TN; ++t)
#pragma unroll
            for (int m = 0; m < MT; ++m) acc[t][m] = make_float2(0.f, 0.f);

        for (int kc = 0; kc < nkc; ++kc, ++j) {
            const int st = j % kStages;
            const uint32_t ph = (j / kStages) & 1;
            const int k0 = kc * kKC + kl;
            const bool active = k0 < a.K;
            uint32_t xh[MT][4];
#pragma unroll
            for (int m = 0; m < MT; ++m) {
                uint4 u = make_uint4(0u, 0u, 0u, 0u);
                if (active && m < M) u = *reinterpret_cast<const uint4 *>(a.X + size_t(m) * a.K + k0);
                xh[m][0] = u.x;
                xh[m][1] = u.y;
                xh[m][2] = u.z;
                xh[m][3] = u.w;
            }
            if (producer) refill(j);
            __syncwarp();
            if (!wbroken && !mbar_wait(&full[st], ph, a.timeout_ns)) wbroken = true;
            if (active && !wbroken) {
                const unsigned char *sp = ring + size_t(st) * SB;
                if (vrows == TN)
                    stage_fma(cuda::std::true_type{}, sp, vrows, xh, acc);
                else
                    stage_fma(cuda::std::false_type{}, sp, vrows, xh, acc);
            }
            __syncwarp();
            if (lane == 0 && !wbroken) mbar_arrive(&empty[st]);
        }

        float vals[NVP];
#pragma unroll
        for (int t = 0; t < TN; ++t)
#pragma unroll
            for (int m = 0; m < MT; ++m) vals[t * MT + m] = acc[t][m].x + acc[t][m].y;
#pragma unroll
        for (int q = NV; q < NVP; ++q) vals[q] = 0.f;
        ReduceScatter<NVP, 16>::run(vals, lane);
        constexpr int LEFT = rs_values_left<NVP, 16>();
        const int first = rs_first_index<NVP, 16>(lane);
#pragma unroll
        for (int q = 0; q < LEFT; ++q) red[warp * NVP + first + q] = vals[q];
        __syncthreads();
        for (int idx = threadIdx.x; idx < NV; idx += kThreadsC) {
            const int t = idx / MT;
            const int m = idx % MT;
            if (t < vrows && m < M) {
                float sum = red[idx];
#pragma unroll
                for (int w = 1; w < kWarpsC; ++w) sum += red[w * NVP + idx];
                const size_t o = size_t(m) * a.N + (n0 + g * TN + t);
                if (a.y_fp32)
                    static_cast<float *>(a.Y)[o] = sum;
                else
                    static_cast<__half *>(a.Y)[o] = __float2half_rn(sum);
            }
        }
        __syncthreads();
    }
}

template <int MT, int TN>
dspark_status launch_ws(const WsArgs &args, int nctas, cudaStream_t stream) {
    auto kern = ws_matvec_kernel<MT, TN>;
    const size_t smem = ws_smem_bytes<TN>(MT);
    static int configured_dev = -1;
    int dev = 0;
    cudaGetDevice(&dev);
    if (configured_dev != dev) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
        if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute(ws_matvec)");
        int per_sm = 0;
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kThreads, smem);
        if (e != cudaSuccess) return cuda_fail(e, "cudaOccupancyMaxActiveBlocksPerMultiprocessor(ws_matvec)");
        if (per_sm < 1) return fail(DSPARK_ERR_CUDA, "ws_matvec kernel cannot be resident on an SM");
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
    args.timeout_ns = kDefaultTimeoutNs;
    const int nctas = N < sms ? N : sms;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    switch (M) {
        case 1: return launch_ws<1, 8>(args, nctas, s);
        case 2: return launch_ws<2, 8>(args, nctas, s);
        case 3: return launch_ws<3, 8>(args, nctas, s);
        case 4: return launch_ws<4, 8>(args, nctas, s);
        case 5: return launch_ws<5, 8>(args, nctas, s);
        case 6: return launch_ws<6, 8>(args, nctas, s);
        case 7: return launch_ws<7, 8>(args, nctas, s);
        case 8: return launch_ws<8, 8>(args, nctas, s);
        default: return launch_ws<16, 2>(args, nctas, s);
    }
}
