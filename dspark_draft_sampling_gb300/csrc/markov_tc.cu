// Markov block draft with the bias GEMV on tcgen05 tensor cores.
//
// Method (vllm.cpp issue #436 "SPEC-DSPARK W7", section "The fix"): per draft position,
// gather markov_w1[prev], bias GEMV over the whole bf16 markov_w2 [vocab, rank], add the
// position's base-logit row, greedy argmax with lowest-index tie-break, d2t map, prev kept
// on the device.
//
// The bias of one vocab row for all requests is the row of markov_w2 times the matrix
// H = [markov_w1[prev_0]; ...; markov_w1[prev_{B-1}]]: a [vocab x rank] x [rank x B] product.
// Here it runs on the 5th-generation tensor cores; the SMs only stream markov_w2 and do the
// argmax epilogue, so the cost no longer grows with the number of requests.
//
// GB300 design (one persistent cooperative launch, one CTA per SM at most)
//  * CTA c owns a contiguous range of 128-row tiles of markov_w2 for every position; odd
//    positions walk it backwards so each position starts on rows still in L2.  The grid is
//    the fewest CTAs that give no CTA more tiles than an even split over all SMs would.
//  * Warp 4 (one thread): per tile, one 3-D TMA tensor copy of the whole [128 rows x rank]
//    bf16 tile (64 KB at rank 256: rank/64 blocks of [128 x 64] in the 128-byte swizzle) and
//    one of the tile's base-logit rows for every request ([num_reqs x 128] fp32) into the same
//    ring slot.  Neither depends on prev, so the producer runs ahead across positions.
//  * Warp 5 allocates 32 TMEM columns (two 128 x 16 fp32 accumulators).  Warps 5 and 6 each
//    have one thread issuing the MMAs of every other tile into its own accumulator: per tile
//    rank/16 tcgen05.mma kind::f16 (bf16 in, fp32 accumulate; M = 128 rows, N = 16 request
//    slots, K = 16) against H, which the epilogue warps write into shared memory in the same
//    swizzled layout (rows >= num_reqs stay zero), then one tcgen05.commit for the slot and
//    one for the accumulator.  Issuing a tile's MMAs takes a good part of a slot's cycle, so
//    two issuers keep tiles that land together from queueing behind one thread.
//  * Warps 0-3 (thread = TMEM lane = vocab row of the tile): read the tile's base logits
//    from the slot as soon as it lands (the slot is free again once both they and the MMAs
//    are done with it), tcgen05.ld the accumulator, keep the best (value, row) per request;
//    at the end of a position turn them into 64-bit keys and reduce (warp, shared atomicMax,
//    one global atomicMax per request), pass the grid barrier, read the winners, write
//    out_ids / prev and build the next position's H from markov_w1.
// Products of bf16 values are exact in fp32; the tensor core accumulates in fp32.  Every
// row's sum is computed the same way regardless of the grid and of num_reqs.
#include <cmath>

#include "markov.cuh"
#include "tc.cuh"

namespace dspark {
namespace {

constexpr int kMmaIssuers = 2;  // issuer p takes the tiles with counter tc % 2 == p (accumulator p)
constexpr int kThreads = 32 * (5 + kMmaIssuers);  // warps 0-3 epilogue, 4 TMA, 5 MMA + TMEM, 6 MMA
constexpr int kEpiThreads = 128;
constexpr int kEpiWarps = kEpiThreads / 32;
constexpr int kTileRows = 128;
constexpr int kKB = 64;                          // k per box (128 B of bf16)
constexpr int kBoxBytes = kTileRows * kKB * 2;   // 16 KB: one 64-k block of a tile
constexpr int kRingBudget = 204 * 1024;          // tile slots: markov_w2 tile + its base rows
constexpr int kMaxSlots = 12;
constexpr int kNPad = 16;                        // MMA N: request slots
constexpr int kHBlockBytes = kNPad * kKB * 2;    // 2 KB per k-block of H
constexpr int kHMaxBytes = 4 * kHBlockBytes;     // rank <= 256
constexpr uint32_t kTmemCols = 32;
constexpr size_t kSmemBytes = 1024 + size_t(kRingBudget) + 2 * kHMaxBytes + 768;
static_assert(kSmemBytes <= 227 * 1024, "shared memory");

// Bytes reserved in a slot for the base rows of NB requests (a multiple of 1024, so the next
// slot's markov_w2 blocks stay aligned for the 128-byte swizzle).
template <int NB>
constexpr int base_area_bytes() {
    return (NB * kTileRows * 4 + 1023) / 1024 * 1024;
}

template <int NB, bool DBG>
__global__ void __launch_bounds__(kThreads, 1)
    markov_tc_kernel(const __grid_constant__ CUtensorMap tmW2, const __grid_constant__ CUtensorMap tmBase,
                     MarkovArgs a, int R, int base_tma) {
    extern __shared__ unsigned char smem_raw[];
    const uint32_t raw = smem_addr(smem_raw);
    unsigned char *smem = smem_raw + ((1024u - (raw & 1023u)) & 1023u);
    unsigned char *ring = smem;
    unsigned char *hbuf = smem + size_t(kRingBudget);  // 2 buffers
    // full[s]: slot s landed (tile and base rows).  empty[s]: the MMAs of the tile in slot s
    // are done (one tcgen05.commit) and the four epilogue warps have read its base rows: the
    // slot may be refilled.  acc_full[b]: accumulator b holds a finished tile (a commit).
    // acc_empty[b]: the epilogue has read accumulator b.
    uint64_t *full = reinterpret_cast<uint64_t *>(hbuf + 2 * kHMaxBytes);
    uint64_t *empty = full + kMaxSlots;
    uint64_t *acc_full = empty + kMaxSlots;  // [2]
    uint64_t *acc_empty = acc_full + 2;      // [2]
    uint64_t *h_full = acc_empty + 2;        // [2]
    unsigned long long *s_best = reinterpret_cast<unsigned long long *>(h_full + 2);  // [kMaxReqs]
    unsigned long long *s_wbest = s_best + kMaxReqs;  // [kEpiWarps][kMaxReqs] each warp's best keys
    int *s_cur = reinterpret_cast<int *>(s_wbest + kEpiWarps * kMaxReqs);            // [kMaxReqs]
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(s_cur + kMaxReqs);
    int *s_abort = reinterpret_cast<int *>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int nctas = gridDim.x;
    const int cta = blockIdx.x;
    const int nkb = R / kKB;
    const int w2_bytes = nkb * kBoxBytes;
    const int slot_bytes = w2_bytes + base_area_bytes<NB>();
    const int nslots = min(kMaxSlots, kRingBudget / slot_bytes);
    const int T = (a.V + kTileRows - 1) / kTileRows;
    // 32-bit unsigned: cta <= 152 and T < 2^24, so cta * T < 2^32
    const int t0 = static_cast<int>(static_cast<unsigned>(cta) * static_cast<unsigned>(T) / static_cast<unsigned>(nctas));
    const int t1 =
        static_cast<int>(static_cast<unsigned>(cta + 1) * static_cast<unsigned>(T) / static_cast<unsigned>(nctas));
    const int ntiles = t1 - t0;
    auto tile_at = [t0, ntiles](int i, int t) { return t0 + ((i & 1) ? ntiles - 1 - t : t); };

    // requests with an out-of-range prev give -1 ids and no candidates
    unsigned bad_mask = 0;
    for (int r = 0; r < a.B; ++r) {
        const long long p = a.prev[r];
        if (p < 0 || p >= a.V) bad_mask |= 1u << r;
    }

    if (threadIdx.x == 0) {
        for (int s = 0; s < kMaxSlots; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1 + kEpiWarps);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&acc_full[b], 1);
            mbar_init(&acc_empty[b], kEpiWarps);
            mbar_init(&h_full[b], kEpiThreads);
        }
        for (int r = 0; r < kMaxReqs; ++r) {
            s_best[r] = 0ull;
            const long long p = r < a.B ? a.prev[r] : 0;
            s_cur[r] = (p >= 0 && p < a.V) ? static_cast<int>(p) : 0;
        }
        *s_abort = 0;
        if (bad_mask && cta == 0) atomicOr(a.status, kStatusIndex);
        fence_mbar_init();
    }
    {  // zero both H buffers (rows >= num_reqs stay zero for the whole kernel)
        uint4 *h4 = reinterpret_cast<uint4 *>(hbuf);
        for (int q = threadIdx.x; q < 2 * kHMaxBytes / 16; q += kThreads) h4[q] = make_uint4(0u, 0u, 0u, 0u);
        fence_proxy_async_smem();
    }
    if (warp == 5) tmem_alloc(tmem_slot, kTmemCols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    // A kernel launched after this one with programmatic dependent launch may start its
    // prologue now; it reads and writes global memory only after this grid has completed.
    pdl_launch_dependents();

    if (warp == 4) {
        // ---------------- TMA producer ----------------
        if (lane == 0) {
            uint64_t pol;
            asm volatile("createpolicy.fractional.L2::evict_normal.b64 %0, 1.0;" : "=l"(pol));
            const uint64_t pol_base = l2_policy_evict_first();
            const uint32_t tx = static_cast<uint32_t>(w2_bytes + (base_tma ? a.B * kTileRows * 4 : 0));
            int st = 0;
            uint32_t ph = 0;
            for (int i = 0; i < a.k; ++i)
                for (int t = 0; t < ntiles; ++t) {
                    const int y = tile_at(i, t) * kTileRows;
                    if (!mbar_wait(&empty[st], ph ^ 1u, a.timeout_ns)) {
                        atomicOr(a.status, kStatusTimeout);
                        goto producer_done;
                    }
                    unsigned char *slot = ring + size_t(st) * slot_bytes;
                    mbar_arrive_expect_tx(&full[st], tx);
                    tma_load_3d(slot, &tmW2, 0, y, 0, &full[st], pol);  // whole tile
                    if (base_tma) tma_load_3d(slot + w2_bytes, &tmBase, y, i, 0, &full[st], pol_base);
                    if (++st == nslots) {
                        st = 0;
                        ph ^= 1u;
                    }
                }
        producer_done:;
        }
    } else if (warp >= 5) {
        // ---------------- MMA issuers: issuer p takes the tiles tc with tc % 2 == p ----------------
        if (lane == 0) {
            const int p = warp - 5;
            constexpr uint32_t idesc = idesc_f16(true, kTileRows, kNPad);
            // Descriptors are built once and advanced by adding byte offsets >> 4 to their
            // address field (all of shared memory is below 256 KB, so it never carries).
            const uint64_t dA0 = smem_desc_sw128(smem_addr(ring));
            const uint64_t dH0 = smem_desc_sw128(smem_addr(hbuf));
            const uint32_t d = tmem + static_cast<uint32_t>(p * kNPad);  // accumulator p
            int tc = 0;
            bool broken = false;
            for (int i = 0; i < a.k && !broken; ++i) {
                // every issuer waits for every position's H, so its parity waits stay exact
                if (!mbar_wait(&h_full[i & 1], (i >> 1) & 1, a.timeout_ns)) {
                    broken = true;
                    break;
                }
                tc_fence_after();
                const uint64_t dH = dH0 + static_cast<uint64_t>((i & 1) * (kHMaxBytes >> 4));
                for (int t = 0; t < ntiles && !broken; ++t, ++tc) {
                    if ((tc & 1) != p) continue;
                    const int st = tc % nslots;
                    const uint32_t ph = static_cast<uint32_t>((tc / nslots) & 1);
                    const uint32_t aph = static_cast<uint32_t>((tc >> 1) & 1);  // use tc / 2 of accumulator p
                    if (!mbar_wait(&acc_empty[p], aph ^ 1u, a.timeout_ns)) {
                        broken = true;
                        break;
                    }
                    if (!mbar_wait(&full[st], ph, a.timeout_ns)) {
                        broken = true;
                        break;
                    }
                    tc_fence_after();
                    const uint64_t dT = dA0 + static_cast<uint64_t>(st * (slot_bytes >> 4));
                    for (int kb = 0; kb < nkb; ++kb) {
                        const uint64_t dA = dT + static_cast<uint64_t>(kb * (kBoxBytes >> 4));
                        const uint64_t dB = dH + static_cast<uint64_t>(kb * (kHBlockBytes >> 4));
                        tc_mma_f16(d, dA, dB, idesc, kb != 0);  // K = 16 per MMA, 32 B apart
                        tc_mma_f16(d, dA + 2, dB + 2, idesc, 1u);
                        tc_mma_f16(d, dA + 4, dB + 4, idesc, 1u);
                        tc_mma_f16(d, dA + 6, dB + 6, idesc, 1u);
                    }
                    tc_commit(&empty[st]);    // the MMAs no longer read the slot
                    tc_commit(&acc_full[p]);  // the accumulator holds the tile
                }
            }
            if (broken) atomicOr(a.status, kStatusTimeout);
        }
    } else {
        // ---------------- epilogue warps: thread = TMEM lane = row of the tile ----------------
        const int et = threadIdx.x;
        auto build_h = [&](int buf) {
            unsigned char *H = hbuf + buf * kHMaxBytes;
            const int cpr = R / 8;  // 16-byte chunks per row
            for (int q = et; q < a.B * cpr; q += kEpiThreads) {
                const int r = q / cpr;
                const int c = q - r * cpr;
                uint4 val = make_uint4(0u, 0u, 0u, 0u);
                if (!((bad_mask >> r) & 1u))
                    val = *reinterpret_cast<const uint4 *>(a.w1 + size_t(s_cur[r]) * R + c * 8);
                const int kb = c >> 3, cc = c & 7;
                *reinterpret_cast<uint4 *>(H + kb * kHBlockBytes + r * 128 + ((cc ^ (r & 7)) << 4)) = val;
            }
            fence_proxy_async_smem();
        };
        build_h(0);
        mbar_arrive(&h_full[0]);

        const unsigned live = (a.B >= 32 ? 0xffffffffu : ((1u << a.B) - 1u)) & ~bad_mask;
        bool aborted = false;  // CTA-uniform: no more computing or grid barriers, keep draining
        bool broken = false;   // one of this thread's waits timed out
        auto give_up = [&]() {
            broken = true;
            atomicOr(a.status, kStatusTimeout);
            *reinterpret_cast<volatile int *>(s_abort) = 1;
        };
        int tc = 0;
        int es = 0;  // slot of tile tc, and the phase of its barriers
        uint32_t eph = 0;
        for (int i = 0; i < a.k; ++i) {
            // best (value, row) per request over this thread's rows; rows are visited in
            // increasing order on even positions and decreasing order on odd ones, so the
            // lowest row among equal values is kept by > and >= respectively
            float bval[NB];
            int bidx[NB];
#pragma unroll
            for (int r = 0; r < NB; ++r) {
                bval[r] = -INFINITY;
                bidx[r] = -1;
            }
            const bool odd = (i & 1) != 0;
            for (int t = 0; t < ntiles; ++t, ++tc) {
                const int ab = tc & 1;
                const uint32_t abph = static_cast<uint32_t>(tc >> 1) & 1u;
                const int row = tile_at(i, t) * kTileRows + et;
                const bool valid = row < a.V && !aborted;
                // the slot's base rows, read as soon as it lands
                if (!broken && !mbar_wait(&full[es], eph, a.timeout_ns)) give_up();
                float bv[NB];
                if (base_tma) {
                    const float *sb = reinterpret_cast<const float *>(ring + size_t(es) * slot_bytes + w2_bytes);
#pragma unroll
                    for (int r = 0; r < NB; ++r) bv[r] = r < a.B ? sb[r * kTileRows + et] : 0.f;
                } else {
#pragma unroll
                    for (int r = 0; r < NB; ++r)
                        bv[r] = (r < a.B && row < a.V) ? __ldg(a.base + (size_t(r) * a.k + i) * a.V + row) : 0.f;
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(&empty[es]);
                if (++es == nslots) {
                    es = 0;
                    eph ^= 1u;
                }
                if (!broken && !mbar_wait(&acc_full[ab], abph, a.timeout_ns)) give_up();
                tc_fence_after();
                uint32_t v[8];
                tmem_ld_8(tmem + ab * kNPad + (static_cast<uint32_t>(warp * 32) << 16), v);
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&acc_empty[ab]);
                if (valid && !broken) {
#pragma unroll
                    for (int r = 0; r < NB; ++r) {
                        if ((live >> r) & 1u) {
                            const float bias = __uint_as_float(v[r]);
                            const float logit = bv[r] + bias;
                            const bool take = bidx[r] < 0 || (odd ? logit >= bval[r] : logit > bval[r]);
                            bval[r] = take ? logit : bval[r];
                            bidx[r] = take ? row : bidx[r];
                            if constexpr (DBG) {
                                const size_t o = (size_t(r) * a.k + i) * a.V + row;
                                if (a.dbg_logits) a.dbg_logits[o] = logit;
                                if (a.dbg_bias) a.dbg_bias[o] = bias;
                            }
                        }
                    }
                }
            }
            if (!aborted) {
                // ---- end of position: CTA max, global max, grid barrier, winner ----
#pragma unroll
                for (int r = 0; r < NB; ++r) {
                    const unsigned long long key =
                        bidx[r] >= 0 ? argmax_key(bval[r], static_cast<uint32_t>(bidx[r])) : 0ull;
                    const unsigned long long k_w = warp_max_u64(key);
                    if (lane == 0) s_wbest[warp * kMaxReqs + r] = k_w;
                }
                named_bar_sync(1, kEpiThreads);
                if (et < a.B) {  // the CTA's best key of request et: the max over the four warps
                    unsigned long long k_c = s_wbest[et];
#pragma unroll
                    for (int w = 1; w < kEpiWarps; ++w) {
                        const unsigned long long k_w = s_wbest[w * kMaxReqs + et];
                        k_c = k_w > k_c ? k_w : k_c;
                    }
                    s_best[et] = k_c;
                }
                named_bar_sync(1, kEpiThreads);
                // A wait of this CTA gave up during the position: its keys miss tiles, so it
                // neither contributes them nor arrives.  The other CTAs' barrier waits then run
                // out too, and no id of this or a later position is written.
                const bool self_broken = *reinterpret_cast<volatile int *>(s_abort) != 0;
                if (!self_broken && et < a.B && s_best[et] != 0ull && i + 1 < a.k) {
                    // this CTA's candidate may be the winner: pull its markov_w1 row into L2 so
                    // the gather after the barrier is an L2 hit
                    const uint32_t cand = argmax_key_index(s_best[et]);
                    const uint16_t *row = a.w1 + size_t(cand) * R;
                    for (int off = 0; off < R * 2; off += 128)
                        asm volatile("prefetch.global.L2::evict_last [%0];" ::"l"(reinterpret_cast<const char *>(row) + off));
                }
                if (et == 0 && !self_broken) {
                    for (int r = 0; r < a.B; ++r) {
                        const unsigned long long k_cta = s_best[r];
                        if (k_cta != 0ull) atomicMax(&a.best[size_t(i) * kMaxReqs + r], k_cta);
                        s_best[r] = 0ull;
                    }
                    // the release orders this thread's atomicMax updates before the arrival
                    red_release_add_u32(a.bar_count, 1u);
                    const unsigned target =
                        static_cast<unsigned>(nctas) * static_cast<unsigned>(i + 1) + a.bar_extra;
                    unsigned spins = 0;
                    unsigned long long ts = 0;
                    while (ld_acquire_u32(a.bar_count) < target) {
                        if (++spins > 256) {
                            if (ts == 0) ts = global_timer_ns();
                            if (global_timer_ns() - ts > a.timeout_ns) {
                                atomicOr(a.status, kStatusTimeout);
                                *reinterpret_cast<volatile int *>(s_abort) = 1;
                                break;
                            }
                            __nanosleep(32);
                        }
                    }
                    // the acquire load above orders the winners' reads after every arrival
                }
                named_bar_sync(1, kEpiThreads);
                if (*reinterpret_cast<volatile int *>(s_abort)) aborted = true;
                if (!aborted && et < a.B && !((bad_mask >> et) & 1u)) {
                    const unsigned long long key = ld_relaxed_u64(&a.best[size_t(i) * kMaxReqs + et]);
                    s_cur[et] = key ? static_cast<int>(argmax_key_index(key)) : 0;
                }
                named_bar_sync(1, kEpiThreads);
                if (!aborted && cta == 0 && et < a.B) {
                    long long out = -1;
                    if (!((bad_mask >> et) & 1u)) {
                        const int id = s_cur[et];
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
                        if (i == a.k - 1) a.prev[et] = id;
                    }
                    a.out_ids[size_t(et) * a.k + i] = out;
                }
            }
            if (i + 1 < a.k) {
                if (!aborted) build_h((i + 1) & 1);
                mbar_arrive(&h_full[(i + 1) & 1]);
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 5) tmem_dealloc(tmem, kTmemCols);
}

template <int NB, bool DBG>
dspark_status launch_nb(const CUtensorMap &tm, const CUtensorMap &tb, const MarkovArgs &args, int R, int base_tma,
                        int nctas, cudaStream_t stream) {
    auto kern = markov_tc_kernel<NB, DBG>;
    static int configured_dev = -1;
    int dev = 0;
    cudaGetDevice(&dev);
    if (configured_dev != dev) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             static_cast<int>(kSmemBytes));
        if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute(markov_tc)");
        int per_sm = 0;
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kThreads, kSmemBytes);
        if (e != cudaSuccess) return cuda_fail(e, "cudaOccupancyMaxActiveBlocksPerMultiprocessor(markov_tc)");
        if (per_sm < 1) return fail(DSPARK_ERR_CUDA, "markov_tc kernel cannot be resident on an SM");
        configured_dev = dev;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(nctas));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = kSmemBytes;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t e = cudaLaunchKernelEx(&cfg, kern, tm, tb, args, R, base_tma);
    if (e != cudaSuccess) return cuda_fail(e, "cudaLaunchKernelEx(markov_tc)");
    return DSPARK_OK;
}

template <bool DBG>
dspark_status launch_dbg(const CUtensorMap &tm, const CUtensorMap &tb, const MarkovArgs &args, int R, int base_tma,
                         int nctas, cudaStream_t stream) {
    if (args.B <= 1) return launch_nb<1, DBG>(tm, tb, args, R, base_tma, nctas, stream);
    if (args.B <= 2) return launch_nb<2, DBG>(tm, tb, args, R, base_tma, nctas, stream);
    if (args.B <= 4) return launch_nb<4, DBG>(tm, tb, args, R, base_tma, nctas, stream);
    return launch_nb<8, DBG>(tm, tb, args, R, base_tma, nctas, stream);
}

}  // namespace

int markov_grid(int V, int sms) {
    const int T = (V + kTileRows - 1) / kTileRows;
    const int per = (T + sms - 1) / sms;  // most tiles any CTA gets with all SMs in use
    return (T + per - 1) / per;           // the fewest CTAs that keep that maximum
}

dspark_status launch_markov_tc(const MarkovArgs &args, int R, int nctas, cudaStream_t stream) {
    if (R % kKB != 0 || R > 256) return fail(DSPARK_ERR_UNSUPPORTED, "markov_tc: rank %d", R);
    CUtensorMap tm, tb;
    dspark_status st = make_tmap_kblocks(&tm, args.w2, true, static_cast<uint64_t>(args.V), static_cast<uint64_t>(R),
                                         kTileRows, static_cast<uint32_t>(R / kKB));
    if (st != DSPARK_OK) return st;
    // base rows by TMA when the tensor map can describe them (row stride a multiple of 16
    // bytes, 16-byte aligned base); otherwise the epilogue loads them itself
    const int base_tma = (args.V % 4 == 0 && aligned(args.base, 16)) ? 1 : 0;
    if (base_tma) {
        st = make_tmap_rows_f32(&tb, args.base, static_cast<uint64_t>(args.B), static_cast<uint64_t>(args.k),
                                static_cast<uint64_t>(args.V), static_cast<uint32_t>(args.B), kTileRows);
        if (st != DSPARK_OK) return st;
    } else {
        tb = tm;  // unused
    }
    if (args.dbg_logits || args.dbg_bias) return launch_dbg<true>(tm, tb, args, R, base_tma, nctas, stream);
    return launch_dbg<false>(tm, tb, args, R, base_tma, nctas, stream);
}

}  // namespace dspark
