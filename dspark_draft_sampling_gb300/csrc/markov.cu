// Markov block-draft sampler: all k draft positions in one persistent cooperative kernel.
//
// Method (vllm.cpp issue #436 "SPEC-DSPARK W7", section "The fix"): per position,
// gather markov_w1[prev], bias GEMV over the whole bf16 markov_w2 [vocab, rank], add the
// position's base-logit row, greedy argmax with lowest-index tie-break, d2t map, and
// carry prev on the device; only the final [num_reqs, k] ids leave the GPU.
//
// GB300 design
//  * One CTA per SM, each owning a fixed contiguous slice of vocab rows for every step.
//  * A producer warp streams the slice's markov_w2 rows through a 7-stage ring of
//    28 KB shared-memory tiles with 1-D TMA bulk copies (cp.async.bulk + mbarrier).
//    markov_w2 does not depend on prev, so the producer runs ahead across step
//    boundaries and HBM stays busy while the consumers wait for the step's argmax.
//  * Seven consumer warps hold h = markov_w1[prev] in registers (fp32, exact from bf16)
//    and evaluate rows with packed fp32x2 FMAs; row sums use a fixed butterfly
//    (reduce-scatter across the lanes of a row), so every logit is produced in one
//    order, independent of grid size and num_reqs.
//  * Argmax candidates are 64-bit keys (order-preserving float code, inverted index):
//    the max key is the greedy argmax with the lowest-index tie-break.  Keys are
//    reduced per CTA with shared-memory atomicMax and across CTAs with one global
//    atomicMax per request: integer max is exact and order-independent, so the result
//    is deterministic (no floating-point atomics anywhere).
//  * A grid-wide barrier (monotonic arrival counter, bounded spin) separates steps;
//    every CTA then reads the winning key, CTA 0 writes out_ids (through d2t) and, at
//    the last step, prev.
#include <cuda/std/type_traits>
#include <cuda_fp16.h>

#include <new>

#include "common.cuh"

namespace dspark {
namespace {

// 1 producer + 7 consumer warps: 8 warps = 2 per SM sub-partition, so each thread may
// hold up to 255 registers (a 9th warp would put 3 warps on one 16K-register partition).
constexpr int kConsumerWarps = 7;
constexpr int kConsumerThreads = kConsumerWarps * 32;
constexpr int kThreads = kConsumerThreads + 32;  // + one producer warp
constexpr int kStages = 7;
constexpr int kTileBytes = 28672;  // 7 x 4 KB: passes divide evenly over 7 warps
constexpr int kMaxReqs = 8;
constexpr size_t kHeaderBytes = 256;  // [0] barrier arrivals, [1] status bits

struct MarkovArgs {
    const float *base;
    const uint16_t *w1;
    const uint16_t *w2;
    const int32_t *d2t;
    int64_t *prev;
    int64_t *out_ids;
    float *dbg_logits;
    float *dbg_bias;
    unsigned *bar_count;
    unsigned *status;
    unsigned long long *best;  // [k][kMaxReqs] winning keys
    int B, k, V;
    unsigned bar_extra;
    unsigned long long timeout_ns;
};

template <int R, int NB>
struct Geo {
    static constexpr int LPR = R >= 256 ? 32 : R / 8;  // lanes per row (16 B each per chunk)
    static constexpr int CH = R / (LPR * 8);           // 16-byte chunks per lane per row
    static constexpr int SLOTS = 32 / LPR;             // rows side by side in one warp
    static constexpr int cmin(int a, int b) { return a < b ? a : b; }
    static constexpr int U = cmin(cmin(8, LPR / NB), 16 / NB);  // rows per slot per pass
    static constexpr int VALS = U * NB;                // sums reduced per lane per pass
    static constexpr int P = SLOTS * U;                // rows per pass
    static constexpr int TR = kTileBytes / (2 * R);    // rows per tile
    static constexpr int PASSES = TR / P;
    static constexpr int PPW = PASSES / kConsumerWarps;  // passes per warp per tile
    static_assert(U >= 1 && VALS <= LPR, "bad geometry");
    static_assert(TR % P == 0 && PASSES % kConsumerWarps == 0 && PPW >= 1, "bad tiling");
};

constexpr size_t smem_bytes() {
    return size_t(kStages) * kTileBytes + 2 * kStages * sizeof(uint64_t) + kMaxReqs * sizeof(unsigned long long) +
           16;
}

template <int R, int NB, bool DBG>
__global__ void __launch_bounds__(kThreads, 1) markov_draft_kernel(MarkovArgs a) {
    using G = Geo<R, NB>;
    extern __shared__ __align__(128) unsigned char smem[];
    unsigned char *ring = smem;
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + size_t(kStages) * kTileBytes);
    uint64_t *empty = full + kStages;
    unsigned long long *s_best = reinterpret_cast<unsigned long long *>(empty + kStages);
    int *s_abort = reinterpret_cast<int *>(s_best + kMaxReqs);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int nctas = gridDim.x;
    const int cta = blockIdx.x;
    const int v0 = static_cast<int>(static_cast<long long>(cta) * a.V / nctas);
    const int v1 = static_cast<int>(static_cast<long long>(cta + 1) * a.V / nctas);
    const int rows_c = v1 - v0;
    const int ntiles = (rows_c + G::TR - 1) / G::TR;
    // Odd positions walk the slice backwards, so each position starts on the rows the
    // previous one touched last -- the ones most likely still in L2.
    auto tile_at = [ntiles](int i, int t) { return (i & 1) ? ntiles - 1 - t : t; };

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], kConsumerWarps);
        }
        for (int r = 0; r < kMaxReqs; ++r) s_best[r] = 0ull;
        *s_abort = 0;
        fence_mbar_init();
    }
    __syncthreads();

    // ---------------- producer warp: stream markov_w2 tiles for every position ---------
    if (warp == kConsumerWarps) {
        if (lane == 0) {
            uint64_t pol;
            asm volatile("createpolicy.fractional.L2::evict_normal.b64 %0, 1.0;" : "=l"(pol));
            int stage = 0;
            uint32_t phase = 0;
            for (int i = 0; i < a.k; ++i) {
                for (int t = 0; t < ntiles; ++t) {
                    if (!mbar_wait(&empty[stage], phase ^ 1u, a.timeout_ns)) {
                        atomicOr(a.status, kStatusTimeout);
                        return;
                    }
                    const int tt = tile_at(i, t);
                    const int rows = min(G::TR, rows_c - tt * G::TR);
                    const uint32_t bytes = static_cast<uint32_t>(rows) * R * 2u;
                    mbar_arrive_expect_tx(&full[stage], bytes);
                    bulk_g2s(ring + size_t(stage) * kTileBytes, a.w2 + size_t(v0 + tt * G::TR) * R, bytes,
                             &full[stage], pol);
                    if (++stage == kStages) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
        }
        return;
    }

    // ---------------- consumer warps ----------------------------------------------------
    const int q = lane % G::LPR;  // sub-lane within a row
    const int slot = lane / G::LPR;
    const int vi = rs_first_index<G::VALS, G::LPR / 2>(lane);
    const int my_u = vi / NB;
    const int my_req = vi % NB;

    // Requests with an out-of-range prev produce -1 ids and no candidates.
    unsigned bad_mask = 0;
    int cur[NB];
#pragma unroll
    for (int r = 0; r < NB; ++r) {
        cur[r] = 0;
        if (r < a.B) {
            const long long p = a.prev[r];
            if (p < 0 || p >= a.V) {
                bad_mask |= 1u << r;
            } else {
                cur[r] = static_cast<int>(p);
            }
        }
    }
    if (bad_mask && cta == 0 && threadIdx.x == 0) atomicOr(a.status, kStatusIndex);
    const bool my_ok = my_req < a.B && !((bad_mask >> my_req) & 1u);

    float2 h2[NB][G::CH][4];
    auto load_h = [&]() {
#pragma unroll
        for (int r = 0; r < NB; ++r) {
#pragma unroll
            for (int c = 0; c < G::CH; ++c) {
                uint4 w = make_uint4(0u, 0u, 0u, 0u);
                if (r < a.B && !((bad_mask >> r) & 1u))
                    w = *reinterpret_cast<const uint4 *>(a.w1 + size_t(cur[r]) * R + c * (G::LPR * 8) + q * 8);
                h2[r][c][0] = bf16x2_to_float2(w.x);
                h2[r][c][1] = bf16x2_to_float2(w.y);
                h2[r][c][2] = bf16x2_to_float2(w.z);
                h2[r][c][3] = bf16x2_to_float2(w.w);
            }
        }
    };
    load_h();

    // Base-logit values this lane needs for the t-th tile of position i, one per pass.
    auto load_base = [&](int i, int t, float (&dst)[G::PPW]) {
        const int tt = tile_at(i, t);
        const int tile_rows = min(G::TR, rows_c - tt * G::TR);
        const float *brow = a.base + (size_t(my_req) * a.k + i) * a.V + (v0 + tt * G::TR);
#pragma unroll
        for (int pw = 0; pw < G::PPW; ++pw) {
            const int row = (warp + pw * kConsumerWarps) * G::P + slot * G::U + my_u;
            dst[pw] = (my_ok && row < tile_rows) ? __ldg(brow + row) : 0.f;
        }
    };

    float bnext[G::PPW];
#pragma unroll
    for (int pw = 0; pw < G::PPW; ++pw) bnext[pw] = 0.f;
    if (ntiles > 0 && a.k > 0) load_base(0, 0, bnext);

    // All passes of one tile.  FULL: every row of the tile exists (no row guards).
    auto consume = [&](auto full_tag, const unsigned char *tile, int tile_rows, int vt0, int i,
                       const float (&bcur)[G::PPW], unsigned long long &best) {
        constexpr bool FULL = decltype(full_tag)::value;
#pragma unroll
        for (int pw = 0; pw < G::PPW; ++pw) {
            const int pass = warp + pw * kConsumerWarps;
            if (FULL || pass * G::P < tile_rows) {
                const int row0 = pass * G::P + slot * G::U;
                float2 acc[G::U][NB];
#pragma unroll
                for (int u = 0; u < G::U; ++u)
#pragma unroll
                    for (int r = 0; r < NB; ++r) acc[u][r] = make_float2(0.f, 0.f);
#pragma unroll
                for (int u = 0; u < G::U; ++u) {
#pragma unroll
                    for (int c = 0; c < G::CH; ++c) {
                        const uint4 wv = *reinterpret_cast<const uint4 *>(
                            tile + size_t(row0 + u) * (R * 2) + (c * (G::LPR * 8) + q * 8) * 2);
                        const uint32_t words[4] = {wv.x, wv.y, wv.z, wv.w};
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const float2 wf = bf16x2_to_float2(words[e]);
#pragma unroll
                            for (int r = 0; r < NB; ++r) acc[u][r] = __ffma2_rn(wf, h2[r][c][e], acc[u][r]);
                        }
                    }
                }
                float vals[G::VALS];
#pragma unroll
                for (int u = 0; u < G::U; ++u)
#pragma unroll
                    for (int r = 0; r < NB; ++r) vals[u * NB + r] = acc[u][r].x + acc[u][r].y;
                ReduceScatter<G::VALS, G::LPR / 2>::run(vals, lane);
                const float bias = vals[0];
                const int row = row0 + my_u;
                const bool valid = my_ok && (FULL || row < tile_rows);
                const float logit = bcur[pw] + bias;
                const int v = vt0 + row;
                const unsigned long long key = argmax_key(logit, static_cast<uint32_t>(v));
                best = (valid && key > best) ? key : best;
                if constexpr (DBG) {
                    if (valid) {
                        const size_t o = (size_t(my_req) * a.k + i) * a.V + v;
                        if (a.dbg_logits) a.dbg_logits[o] = logit;
                        if (a.dbg_bias) a.dbg_bias[o] = bias;
                    }
                }
            }
        }
    };

    int stage = 0;
    uint32_t phase = 0;
    // aborted: CTA-uniform (taken from s_abort after a named barrier); the consumers then
    //   stop computing and synchronizing but keep draining the ring so the producer ends.
    // broken: this warp's wait on a tile timed out; it waits on no further tiles but still
    //   reaches every named barrier, so no warp of the CTA is left waiting.
    bool aborted = false;
    bool broken = false;

    for (int i = 0; i < a.k; ++i) {
        unsigned long long best = 0ull;
        for (int t = 0; t < ntiles; ++t) {
            float bcur[G::PPW];
#pragma unroll
            for (int pw = 0; pw < G::PPW; ++pw) bcur[pw] = bnext[pw];
            {
                int ni = i, nt = t + 1;
                if (nt == ntiles) {
                    nt = 0;
                    ++ni;
                }
                if (ni < a.k && !aborted) load_base(ni, nt, bnext);
            }
            if (!broken && !mbar_wait(&full[stage], phase, a.timeout_ns)) {
                if (lane == 0) {
                    atomicOr(a.status, kStatusTimeout);
                    *reinterpret_cast<volatile int *>(s_abort) = 1;
                }
                broken = true;
            }
            if (!aborted && !broken) {
                const int tt = tile_at(i, t);
                const int tile_rows = min(G::TR, rows_c - tt * G::TR);
                const unsigned char *tile = ring + size_t(stage) * kTileBytes;
                if (tile_rows == G::TR)
                    consume(cuda::std::true_type{}, tile, tile_rows, v0 + tt * G::TR, i, bcur, best);
                else
                    consume(cuda::std::false_type{}, tile, tile_rows, v0 + tt * G::TR, i, bcur, best);
            }
            __syncwarp();
            if (lane == 0 && !broken) mbar_arrive(&empty[stage]);
            if (++stage == kStages) {
                stage = 0;
                phase ^= 1u;
            }
        }
        if (aborted) continue;  // keep draining the ring; no more barriers

        // ---- end of position: CTA max, global max, grid barrier, winner ----------------
        if (my_ok && best != 0ull) atomicMax(&s_best[my_req], best);
        named_bar_sync(1, kConsumerThreads);
        if (threadIdx.x == 0) {
            // one thread publishes the CTA's keys, then arrives: its release orders them
            for (int r = 0; r < a.B; ++r) {
                const unsigned long long k_cta = s_best[r];
                if (k_cta != 0ull) atomicMax(&a.best[size_t(i) * kMaxReqs + r], k_cta);
                s_best[r] = 0ull;
            }
            __threadfence();
            red_release_add_u32(a.bar_count, 1u);
            const unsigned target = static_cast<unsigned>(nctas) * static_cast<unsigned>(i + 1) + a.bar_extra;
            unsigned spins = 0;
            unsigned long long t0 = 0;
            while (ld_acquire_u32(a.bar_count) < target) {
                if (++spins > 256) {
                    if (t0 == 0) t0 = global_timer_ns();
                    if (global_timer_ns() - t0 > a.timeout_ns) {
                        atomicOr(a.status, kStatusTimeout);
                        *reinterpret_cast<volatile int *>(s_abort) = 1;
                        break;
                    }
                    __nanosleep(32);
                }
            }
            __threadfence();
        }
        named_bar_sync(1, kConsumerThreads);
        if (*reinterpret_cast<volatile int *>(s_abort)) {
            aborted = true;
            continue;
        }
#pragma unroll
        for (int r = 0; r < NB; ++r) {
            if (r < a.B && !((bad_mask >> r) & 1u)) {
                const unsigned long long key = ld_relaxed_u64(&a.best[size_t(i) * kMaxReqs + r]);
                // every row yields a key > 0, so key 0 cannot win; guard the gather anyway
                cur[r] = key ? static_cast<int>(argmax_key_index(key)) : 0;
            }
        }
        if (i + 1 < a.k) load_h();
        if (cta == 0 && threadIdx.x < a.B) {
            const int r = threadIdx.x;
            long long out = -1;
            if (!((bad_mask >> r) & 1u)) {
                int id = 0;
#pragma unroll
                for (int rr = 0; rr < NB; ++rr)
                    if (rr == r) id = cur[rr];
                out = id;
                if (a.d2t) {
                    const int tgt = a.d2t[id];
                    if (tgt < 0) {
                        out = -1;
                        atomicOr(a.status, kStatusIndex);
                    } else {
                        out = tgt;
                    }
                }
                if (i == a.k - 1) a.prev[r] = id;
            }
            a.out_ids[size_t(r) * a.k + i] = out;
        }
    }
}

template <int R, int NB, bool DBG>
dspark_status launch_markov(const MarkovArgs &args, int nctas, cudaStream_t stream) {
    auto kern = markov_draft_kernel<R, NB, DBG>;
    static bool configured = false;  // per-process: the attribute is set on every device used
    static int configured_dev = -1;
    int dev = 0;
    cudaGetDevice(&dev);
    if (!configured || configured_dev != dev) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             static_cast<int>(smem_bytes()));
        if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute(markov)");
        int per_sm = 0;
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kThreads, smem_bytes());
        if (e != cudaSuccess) return cuda_fail(e, "cudaOccupancyMaxActiveBlocksPerMultiprocessor(markov)");
        if (per_sm < 1) return fail(DSPARK_ERR_CUDA, "markov kernel cannot be resident on an SM");
        configured = true;
        configured_dev = dev;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(nctas));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem_bytes();
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t e = cudaLaunchKernelEx(&cfg, kern, args);
    if (e != cudaSuccess) return cuda_fail(e, "cudaLaunchKernelEx(markov)");
    return DSPARK_OK;
}

template <int R, bool DBG>
dspark_status launch_reqs(const MarkovArgs &args, int nctas, cudaStream_t stream) {
    if (args.B <= 1) return launch_markov<R, 1, DBG>(args, nctas, stream);
    if (args.B <= 2) return launch_markov<R, 2, DBG>(args, nctas, stream);
    if (args.B <= 4) return launch_markov<R, 4, DBG>(args, nctas, stream);
    return launch_markov<R, 8, DBG>(args, nctas, stream);
}

template <int R>
dspark_status launch_rank(const MarkovArgs &args, int nctas, cudaStream_t stream) {
    if (args.dbg_logits || args.dbg_bias) return launch_reqs<R, true>(args, nctas, stream);
    return launch_reqs<R, false>(args, nctas, stream);
}

size_t workspace_bytes(int k) {
    const size_t keys = size_t(k > 0 ? k : 0) * kMaxReqs * sizeof(unsigned long long);
    return (kHeaderBytes + keys + 255) / 256 * 256;
}

dspark_status markov_enqueue(const float *base, const uint16_t *w1, const uint16_t *w2, const int32_t *d2t,
                             int64_t *prev, int B, int k, int V, int R, int64_t *out_ids, float *dbg_logits,
                             float *dbg_bias, void *workspace, size_t ws_bytes, unsigned bar_extra,
                             unsigned long long timeout_ns, cudaStream_t stream) {
    clear_error();
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

    unsigned char *ws = static_cast<unsigned char *>(workspace);
    cudaError_t e = cudaMemsetAsync(ws, 0, workspace_bytes(k), stream);
    if (e != cudaSuccess) return cuda_fail(e, "cudaMemsetAsync(markov workspace)");
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
    switch (R) {
        case 64: return launch_rank<64>(args, sms, stream);
        case 128: return launch_rank<128>(args, sms, stream);
        default: return launch_rank<256>(args, sms, stream);
    }
}

}  // namespace
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
                                  reinterpret_cast<cudaStream_t>(stream));
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
// Device address of the scratch array, looked up once per device with that device current.
dspark_status noalloc_scratch(void **out) {
    static void *addr[64] = {nullptr};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    if (dev < 0 || dev >= 64) return fail(DSPARK_ERR_UNSUPPORTED, "markov_noalloc: device ordinal %d >= 64", dev);
    void *p = __atomic_load_n(&addr[dev], __ATOMIC_ACQUIRE);
    if (!p) {
        e = cudaGetSymbolAddress(&p, g_markov_noalloc_scratch);
        if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(markov scratch)");
        __atomic_store_n(&addr[dev], p, __ATOMIC_RELEASE);
    }
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
    return dspark::markov_enqueue(base_logits, markov_w1, markov_w2, d2t, prev, num_reqs, k, vocab, rank, out_ids,
                                  nullptr, nullptr, scratch, dspark::kNoAllocScratchBytes, 0u,
                                  dspark::kDefaultTimeoutNs, reinterpret_cast<cudaStream_t>(stream));
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
