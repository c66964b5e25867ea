// Markov block draft for small vocabularies: all k positions in one thread-block cluster.
//
// Method (vllm.cpp issue #436 "SPEC-DSPARK W7", section "The fix"): per draft position,
// gather markov_w1[prev], bias GEMV over the whole bf16 markov_w2 [vocab, rank], add the
// position's base-logit row, greedy argmax with lowest-index tie-break, d2t map, prev kept
// on the device.
//
// With a small draft vocabulary the grid-wide form (markov_tc.cu) spends almost all of a
// position on the chain of global-memory round trips that pass the argmax between CTAs.
// When markov_w2 and markov_w1 fit in the shared memory of one cluster of up to 16 CTAs,
// this kernel keeps that chain on chip:
//  * CTA c of the cluster owns a contiguous range of 128-row tiles and loads its tiles of
//    markov_w2 and markov_w1 once, by TMA, in the 128-byte-swizzled [128 x 64] block layout
//    (chunk q of row r of a block at chunk q ^ (r & 7)), and keeps them for all positions.
//    The base-logit rows of each position stream through a ring of buffers, several
//    positions ahead.
//  * Per position the tcgen05 MMAs of the CTA's tiles run against H with the same instruction
//    shape and K order as the grid form (M = 128 rows, N = 16 request slots, K = 16, rank/16
//    MMAs per tile, one fp32 accumulator of 16 TMEM columns per tile), so every bias value is
//    bit-identical to the grid form's.  Warpgroup g (warps 4g .. 4g + 3) takes the tiles
//    j with j % 2 == g: lane 0 of its first warp issues their MMAs from the warpgroup's own
//    copy of H, and its four warps read the accumulators (warp w: TMEM lanes 32 (w % 4) ...),
//    add the base logits and keep the best 64-bit (value, lowest index) key per request.
//  * Exchange without a cluster barrier: per request, the CTA's best key and the markov_w1 row
//    of its candidate go to every CTA of the cluster (itself included) as 16-byte st.async
//    stores straight from registers, whose bytes complete on the receiving CTA's inbox
//    barrier.  The issuing warp of each warpgroup waits only for its own CTA's inbox: the max
//    over the C keys is the winner, its markov_w1 row is already there, so the warp writes its
//    next H and issues its next MMAs while the other warps wait for them.  Inboxes and
//    barriers alternate by position parity; a CTA cannot send position i + 2 before every CTA
//    has sent position i + 1, which each does only after it has read its inbox of position i
//    and armed it again, so two are enough.
//  * CTA 0 records the winners and, after the last position, writes out_ids (through d2t)
//    and prev.  A final cluster barrier keeps every CTA alive until no store to it is in
//    flight.
#include <cmath>

#include "markov.cuh"
#include "tc.cuh"

namespace dspark {
namespace {

constexpr int kThreadsC = 256;
constexpr int kWarpsC = kThreadsC / 32;
constexpr int kTileRowsC = 128;
constexpr int kBlockBytes = kTileRowsC * 64 * 2;  // one [128 x 64] bf16 block of a tile: 16 KB
constexpr int kNPadC = 16;                        // MMA N: request slots (as the grid form)
constexpr int kHBlockBytesC = kNPadC * 128;       // one 64-column block of H: 2 KB
constexpr int kMaxCluster = 16;
constexpr int kMaxBaseBufs = 8;
constexpr size_t kSmemLimit = 227 * 1024;

// Shared-memory layout of one CTA; identical in every CTA of the cluster, so that a location
// in this CTA maps to the same location in a peer by mapa.
struct ClusterLayout {
    size_t w2, w1, h, base, inbox, wkey, ids, bars, flags, tmem_slot, total;
    int tile_bytes;   // one 128-row tile of one matrix: 128 * R * 2
    int base_stride;  // one tile's base rows for NB requests
    int msg;          // one request's message: 8-byte key, 8 bytes of padding, the 2R-byte row
};

__host__ __device__ inline ClusterLayout cluster_layout(int ntile, int R, int NB, int C, int nbuf, int k) {
    ClusterLayout L;
    L.tile_bytes = kTileRowsC * R * 2;
    L.base_stride = NB * kTileRowsC * 4;
    L.msg = 16 + 2 * R;
    size_t o = 0;  // from a 1024-byte aligned base
    L.w2 = o;
    o += size_t(ntile) * L.tile_bytes;
    L.w1 = o;
    o += size_t(ntile) * L.tile_bytes;
    L.h = o;  // [2 warpgroups][R / 64][16 rows][128 B], 128-byte swizzle
    o += size_t(2) * (R / 64) * kHBlockBytesC;
    L.base = o;
    o += size_t(nbuf) * ntile * L.base_stride;
    L.inbox = o;  // [2][C][NB] messages, by position parity and sender
    o += size_t(2) * C * NB * L.msg;
    L.wkey = o;  // u64 [2][kWarpsC][kMaxReqs], by position parity
    o += size_t(2) * kWarpsC * kMaxReqs * 8;
    L.ids = o;  // int [k][kMaxReqs]: the winners, draft space
    o += (size_t(k) * kMaxReqs * 4 + 15) / 16 * 16;
    L.bars = o;  // u64: w2, w1, acc[2], inbox[2], base[kMaxBaseBufs]
    o += (6 + kMaxBaseBufs) * 8;
    L.flags = o;  // int [4]: [0] this CTA gave up, [1] positions done (end of the kernel)
    o += 16;
    L.tmem_slot = o;
    o += 16;
    L.total = 1024 + o;  // slack for aligning the dynamic shared memory to 1024 bytes
    return L;
}

__device__ __forceinline__ uint32_t dsmem_map(uint32_t local_smem_addr, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(local_smem_addr), "r"(rank));
    return r;
}

// 16-byte store into the shared memory of a CTA of the cluster whose bytes complete on the
// barrier `remote_bar` of that CTA (both addresses from mapa).
__device__ __forceinline__ void st_async_v4(uint32_t remote_addr, uint4 v, uint32_t remote_bar) {
    asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.v4.b32 [%0], {%1, %2, %3, %4}, [%5];" ::"r"(
                     remote_addr),
                 "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w), "r"(remote_bar)
                 : "memory");
}

// Every thread of every CTA of the cluster; the warp must be converged (aligned form).
__device__ __forceinline__ void cluster_barrier() {
    __syncwarp();
    asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
    asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// First tile of CTA c when T tiles are split over C CTAs (contiguous, balanced).
__host__ __device__ inline int tile_begin(int c, int T, int C) {
    return static_cast<int>(static_cast<unsigned>(c) * static_cast<unsigned>(T) / static_cast<unsigned>(C));
}

__host__ __device__ inline uint32_t tmem_cols_for(int ntile) {
    uint32_t n = 32;
    while (n < static_cast<uint32_t>(ntile * kNPadC)) n <<= 1;
    return n;
}

template <int NB, bool DBG>
__global__ void __launch_bounds__(kThreadsC, 1)
    markov_cluster_kernel(const __grid_constant__ CUtensorMap tmW2, const __grid_constant__ CUtensorMap tmW1,
                          const __grid_constant__ CUtensorMap tmBase, MarkovArgs a, int R, int nbuf) {
    extern __shared__ unsigned char smem_raw[];
    const uint32_t raw = smem_addr(smem_raw);
    unsigned char *smem = smem_raw + ((1024u - (raw & 1023u)) & 1023u);
    const int C = gridDim.x;  // the whole grid is one cluster
    const int rank = blockIdx.x;
    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;
    const int T = (a.V + kTileRowsC - 1) / kTileRowsC;
    const int t0 = tile_begin(rank, T, C);
    const int ntile = tile_begin(rank + 1, T, C) - t0;
    const int ntile_max = (T + C - 1) / C;
    const ClusterLayout L = cluster_layout(ntile_max, R, NB, C, nbuf, a.k);
    const int nkb = R / 64;
    const int cpr = R / 8;  // 16-byte chunks per row
    const uint32_t tmem_cols = tmem_cols_for(ntile_max);
    // Warpgroup g (warps 4g .. 4g + 3) reads the accumulators of the tiles j with j % 2 == g;
    // lane 0 of warp 4g issues their MMAs from its own copy of H.
    const int wg = warp >> 2;
    const int ngroups = ntile >= 2 ? 2 : 1;
    const bool issuer_warp = (warp & 3) == 0 && wg < ngroups;
    constexpr int kBaseIssuer = kThreadsC - 32;  // lane 0 of the last warp requests the base rows

    unsigned char *w2s = smem + L.w2;
    unsigned char *w1s = smem + L.w1;
    unsigned char *hb = smem + L.h + size_t(wg) * nkb * kHBlockBytesC;  // this warpgroup's H
    unsigned char *inbox = smem + L.inbox;
    unsigned long long *wkey = reinterpret_cast<unsigned long long *>(smem + L.wkey);  // [2][warps][reqs]
    int *s_ids = reinterpret_cast<int *>(smem + L.ids);
    uint64_t *bar_w2 = reinterpret_cast<uint64_t *>(smem + L.bars);
    uint64_t *bar_w1 = bar_w2 + 1;
    uint64_t *bar_acc = bar_w2 + 2;  // [2], one per warpgroup
    uint64_t *bar_in = bar_w2 + 4;   // [2], by position parity
    uint64_t *bar_base = bar_w2 + 6;
    volatile int *flags = reinterpret_cast<volatile int *>(smem + L.flags);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + L.tmem_slot);
    const uint32_t in_tx = static_cast<uint32_t>(C * a.B * L.msg);  // bytes of one position's inbox

    unsigned bad_mask = 0;  // requests whose prev is outside [0, V): ids -1, no candidates
    for (int r = 0; r < a.B; ++r) {
        const long long p = a.prev[r];
        if (p < 0 || p >= a.V) bad_mask |= 1u << r;
    }
    const unsigned live = ((1u << a.B) - 1u) & ~bad_mask;

    // set-up; the matrix tiles and the first positions' base rows are requested first so that
    // everything else overlaps their flight
    const uint32_t base_tx = static_cast<uint32_t>(ntile * a.B * kTileRowsC * 4);
    auto issue_base = [&](int p) {
        const int b = p % nbuf;
        unsigned char *dst = smem + L.base + size_t(b) * ntile_max * L.base_stride;
        mbar_arrive_expect_tx(&bar_base[b], base_tx);
        const uint64_t pol = l2_policy_evict_first();
        for (int j = 0; j < ntile; ++j)
            tma_load_3d(dst + size_t(j) * L.base_stride, &tmBase, (t0 + j) * kTileRowsC, p, 0, &bar_base[b], pol);
    };
    const int nbuf0 = a.k < nbuf ? a.k : nbuf;  // positions requested up front
    int issued = nbuf0;  // positions whose base rows were requested (meaningful in kBaseIssuer)
    if (tid == 0) {
        mbar_init(bar_w2, 1);
        mbar_init(bar_w1, 1);
        for (int g = 0; g < 2; ++g) mbar_init(&bar_acc[g], 1);
        for (int b = 0; b < 2; ++b) mbar_init(&bar_in[b], 1);
        for (int b = 0; b < kMaxBaseBufs; ++b) mbar_init(&bar_base[b], 1);
        fence_mbar_init();
        const uint64_t pol = l2_policy_evict_last();
        mbar_arrive_expect_tx(bar_w2, static_cast<uint32_t>(ntile * L.tile_bytes));
        for (int j = 0; j < ntile; ++j)
            tma_load_3d(w2s + size_t(j) * L.tile_bytes, &tmW2, 0, (t0 + j) * kTileRowsC, 0, bar_w2, pol);
        mbar_arrive_expect_tx(bar_w1, static_cast<uint32_t>(ntile * L.tile_bytes));
        for (int j = 0; j < ntile; ++j)
            tma_load_3d(w1s + size_t(j) * L.tile_bytes, &tmW1, 0, (t0 + j) * kTileRowsC, 0, bar_w1, pol);
        for (int p = 0; p < nbuf0; ++p) issue_base(p);
        // the inboxes of positions 0 and 1 are armed before any CTA can send (cluster barrier)
        mbar_arrive_expect_tx(&bar_in[0], in_tx);
        if (a.k > 1) mbar_arrive_expect_tx(&bar_in[1], in_tx);
        flags[0] = 0;
        flags[1] = 0;
        // The status word belongs to this call from here on: every update to it comes after
        // the cluster barrier below.
        if (rank == 0) *a.status = 0u;
    }
    if (warp == 0) tmem_alloc(tmem_slot, tmem_cols);
    // H of the first position from global memory, in both copies: row r = markov_w1[prev_r]
    // (rows >= num_reqs and requests with a bad prev stay zero), in the MMA's swizzled layout
    for (int q = tid; q < kNPadC * cpr; q += kThreadsC) {
        const int r = q / cpr;
        const int c = q - r * cpr;
        uint4 v = make_uint4(0u, 0u, 0u, 0u);
        if (r < NB && ((live >> r) & 1u)) v = ldg_nc_v4(a.w1 + size_t(a.prev[r]) * R + c * 8);
        const int kb = c >> 3, cc = c & 7;
        const size_t o = size_t(kb) * kHBlockBytesC + r * 128 + ((cc ^ (r & 7)) << 4);
        *reinterpret_cast<uint4 *>(smem + L.h + o) = v;
        *reinterpret_cast<uint4 *>(smem + L.h + size_t(nkb) * kHBlockBytesC + o) = v;
    }
    fence_proxy_async_smem();
    tc_fence_before();
    // Every CTA of the cluster is running, has initialised its barriers and armed its inboxes
    // before any store into it; the status word is reset before any update.
    cluster_barrier();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    if (rank == 0 && tid == 0 && bad_mask) atomicOr(a.status, kStatusIndex);

    auto give_up = [&]() {
        atomicOr(a.status, kStatusTimeout);
        flags[0] = 1;
    };
    constexpr uint32_t idesc = idesc_f16(true, kTileRowsC, kNPadC);
    auto issue_mmas = [&]() {  // this warpgroup's tiles against its H; one commit
        const uint64_t dA0 = smem_desc_sw128(smem_addr(w2s));
        const uint64_t dH0 = smem_desc_sw128(smem_addr(hb));
        for (int j = wg; j < ntile; j += 2) {
            const uint32_t d = tmem + static_cast<uint32_t>(j * kNPadC);
            const uint64_t dT = dA0 + static_cast<uint64_t>((j * L.tile_bytes) >> 4);
            for (int kb = 0; kb < nkb; ++kb) {
                const uint64_t dA = dT + static_cast<uint64_t>(kb * (kBlockBytes >> 4));
                const uint64_t dB = dH0 + static_cast<uint64_t>(kb * (kHBlockBytesC >> 4));
                tc_mma_f16(d, dA, dB, idesc, kb != 0);  // K = 16 per MMA, 32 B apart
                tc_mma_f16(d, dA + 2, dB + 2, idesc, 1u);
                tc_mma_f16(d, dA + 4, dB + 4, idesc, 1u);
                tc_mma_f16(d, dA + 6, dB + 6, idesc, 1u);
            }
        }
        tc_commit(&bar_acc[wg]);
    };
    int mma_issued = 0;  // positions whose MMAs were issued (meaningful in the issuing lanes)
    int done = 0;        // positions whose winners are known (meaningful in warp 0)
    if (issuer_warp && lane == 0) {
        if (mbar_wait(bar_w2, 0, a.timeout_ns)) {
            issue_mmas();
            mma_issued = 1;
        } else {
            give_up();
            mbar_arrive(&bar_acc[wg]);  // release the warpgroup's wait: nothing comes
        }
    }

    const int lane_base = (warp & 3) * 32;    // TMEM lanes (= tile rows) of this warp
    const int items = a.B * (cpr + 1);          // 16-byte pieces of one message: key + row chunks
    int pg = kThreadsC / items;                 // peer groups: threads that send the same piece
    pg = pg < 1 ? 1 : (pg > C ? C : pg);
    // this thread's first piece (the same at every position): peer group, request, chunk
    // (chunk cpr is the key), and the piece's offset within one message
    const int q0g = tid / items;
    const int q0r = (tid - q0g * items) / (cpr + 1);
    const int q0c = tid - q0g * items - q0r * (cpr + 1);
    for (int i = 0; i < a.k; ++i) {
        const int par = i & 1;
        const int b = i % nbuf;
        if (!flags[0] && !mbar_wait(&bar_base[b], static_cast<uint32_t>((i / nbuf) & 1), a.timeout_ns)) give_up();
        if (wg < ngroups && !flags[0] && !mbar_wait(&bar_acc[wg], static_cast<uint32_t>(i & 1), a.timeout_ns))
            give_up();
        // the candidates' markov_w1 rows are sent from the first position on
        if (i == 0 && !flags[0] && !mbar_wait(bar_w1, 0, a.timeout_ns)) give_up();
        tc_fence_after();
        const float *bsm = reinterpret_cast<const float *>(smem + L.base + size_t(b) * ntile_max * L.base_stride);
        unsigned long long key[NB];
#pragma unroll
        for (int r = 0; r < NB; ++r) key[r] = 0ull;
        for (int j = wg; j < ntile; j += 2) {
            uint32_t v[8];
            tmem_ld_8(tmem + j * kNPadC + (static_cast<uint32_t>(lane_base) << 16), v);
            const int rit = lane_base + lane;
            const int row = (t0 + j) * kTileRowsC + rit;
            if (row < a.V && !flags[0]) {
#pragma unroll
                for (int r = 0; r < NB; ++r) {
                    if ((live >> r) & 1u) {
                        const float bias = __uint_as_float(v[r]);
                        const float logit = bsm[j * (NB * kTileRowsC) + r * kTileRowsC + rit] + bias;
                        const unsigned long long kv = argmax_key(logit, static_cast<uint32_t>(row));
                        key[r] = kv > key[r] ? kv : key[r];
                        if constexpr (DBG) {
                            const size_t o = (size_t(r) * a.k + i) * a.V + row;
                            if (a.dbg_logits) a.dbg_logits[o] = logit;
                            if (a.dbg_bias) a.dbg_bias[o] = bias;
                        }
                    }
                }
            }
        }
        unsigned long long *wk = wkey + par * (kWarpsC * kMaxReqs);
#pragma unroll
        for (int r = 0; r < NB; ++r) {
            const unsigned long long kw = warp_max_u64(key[r]);
            if (lane == 0) wk[warp * kMaxReqs + r] = kw;
        }
        tc_fence_before();
        __syncthreads();  // warp keys in; the accumulators and this base buffer are no longer read
        const bool gave_up = flags[0] != 0;
        if (tid == kBaseIssuer && i + nbuf < a.k && !gave_up) {
            issue_base(i + nbuf);
            issued = i + nbuf + 1;
        }
        // send: per request the CTA's best key and the markov_w1 row of its candidate, to every
        // CTA of the cluster (this one included), straight from registers
        if (!gave_up) {
            for (int q = tid; q < items * pg; q += kThreadsC) {
                int g = q0g, r = q0r, c = q0c;
                if (q != tid) {  // more pieces than threads: only with many requests and rank 256
                    g = q / items;
                    const int it = q - g * items;
                    r = it / (cpr + 1);
                    c = it - r * (cpr + 1);
                }
                unsigned long long kc = wk[r];
#pragma unroll
                for (int w = 1; w < kWarpsC; ++w) {
                    const unsigned long long kw = wk[w * kMaxReqs + r];
                    kc = kw > kc ? kw : kc;
                }
                uint4 v = make_uint4(static_cast<uint32_t>(kc), static_cast<uint32_t>(kc >> 32), 0u, 0u);
                if (c < cpr) {
                    v = make_uint4(0u, 0u, 0u, 0u);
                    if (kc != 0ull) {
                        const int lr = static_cast<int>(argmax_key_index(kc)) - t0 * kTileRowsC;  // row in this CTA
                        const int j = lr >> 7, rit = lr & (kTileRowsC - 1);
                        const int kb = c >> 3, cc = c & 7;
                        v = *reinterpret_cast<const uint4 *>(w1s + size_t(j) * L.tile_bytes + kb * kBlockBytes +
                                                             rit * 128 + ((cc ^ (rit & 7)) << 4));
                    }
                }
                const uint32_t loc = smem_addr(inbox) + static_cast<uint32_t>(((par * C + rank) * NB + r) * L.msg +
                                                                              (c < cpr ? 16 + c * 16 : 0));
                const uint32_t bar = smem_addr(&bar_in[par]);
                for (int p = g; p < C; p += pg)
                    st_async_v4(dsmem_map(loc, static_cast<uint32_t>(p)), v, dsmem_map(bar, static_cast<uint32_t>(p)));
            }
        }
        if (issuer_warp) {
            // every CTA's message of position i is in this CTA's inbox: the winners, then this
            // warpgroup's next H and MMAs
            bool ok = !gave_up;
            if (ok && !mbar_wait(&bar_in[par], static_cast<uint32_t>((i >> 1) & 1), a.timeout_ns)) ok = false;
            ok = __all_sync(0xffffffffu, ok);
            // Winners: per request, lane l < C holds sender l's key; the warp max is the
            // winner, the lane holding it its sender.
            int src_of[NB];
#pragma unroll
            for (int r = 0; r < NB; ++r) {
                src_of[r] = -1;
                if (r < a.B) {
                    unsigned long long kv = 0ull;
                    if (ok && lane < C) {
                        const uint2 k2 =
                            *reinterpret_cast<const uint2 *>(inbox + ((size_t(par) * C + lane) * NB + r) * L.msg);
                        kv = (static_cast<unsigned long long>(k2.y) << 32) | k2.x;
                    }
                    const unsigned long long best = warp_max_u64(kv);
                    const unsigned hold = __ballot_sync(0xffffffffu, best != 0ull && kv == best);
                    const bool has = ok && ((live >> r) & 1u) && best != 0ull;
                    if (has) src_of[r] = __ffs(hold) - 1;
                    if (warp == 0 && lane == 0) s_ids[i * kMaxReqs + r] = has ? static_cast<int>(argmax_key_index(best)) : -1;
                }
            }
            if (ok) done = i + 1;
            if (ok && i + 1 < a.k) {
                const int n = a.B * cpr;
                for (int q = lane; q < n; q += 32) {
                    const int r = q / cpr;
                    const int c = q - r * cpr;
                    int sr = -1;
#pragma unroll
                    for (int rr = 0; rr < NB; ++rr)
                        if (rr == r) sr = src_of[rr];
                    {
                        uint4 v = make_uint4(0u, 0u, 0u, 0u);
                        if (sr >= 0)
                            v = *reinterpret_cast<const uint4 *>(inbox + ((size_t(par) * C + sr) * NB + r) * L.msg +
                                                                 16 + c * 16);
                        const int kb = c >> 3, cc = c & 7;
                        *reinterpret_cast<uint4 *>(hb + kb * kHBlockBytesC + r * 128 + ((cc ^ (r & 7)) << 4)) = v;
                    }
                }
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) {
                    // inbox of position i + 2: its senders need this CTA's message of position
                    // i + 1 first, which leaves only after both issuing warps are done with it
                    if (warp == 0 && i + 2 < a.k) mbar_arrive_expect_tx(&bar_in[par], in_tx);
                    tc_fence_after();
                    issue_mmas();
                    ++mma_issued;
                }
            }
            if (!ok && !gave_up && lane == 0) {
                give_up();
                mbar_arrive(&bar_acc[wg]);  // release the warpgroup's wait: no MMA comes
                mma_issued = 0;             // (its last commit was already waited for)
            }
            __syncwarp();
        }
    }
    // The CTA's last position is done; stores sent to it that a wait gave up on, copies and
    // MMAs land before it exits (each wait again with the limit).
    if (flags[0]) {
        if (tid == 0) {
            for (int p = done; p < a.k && p < done + 2; ++p)
                mbar_wait(&bar_in[p & 1], static_cast<uint32_t>((p >> 1) & 1), a.timeout_ns);
            mbar_wait(bar_w2, 0, a.timeout_ns);
            mbar_wait(bar_w1, 0, a.timeout_ns);
        }
        if (issuer_warp && lane == 0 && mma_issued > 0)
            mbar_wait(&bar_acc[wg], static_cast<uint32_t>((mma_issued - 1) & 1), a.timeout_ns);
        if (tid == kBaseIssuer) {  // the last request into each base buffer
            for (int p = issued - 1; p >= 0 && p >= issued - nbuf; --p)
                mbar_wait(&bar_base[p % nbuf], static_cast<uint32_t>((p / nbuf) & 1), a.timeout_ns);
        }
    }
    if (tid == 0) flags[1] = done;
    __syncthreads();
    if (rank == 0) {
        const int nd = flags[1];
        for (int q = tid; q < a.B * nd; q += kThreadsC) {
            const int r = q / nd;
            const int i = q - r * nd;
            const int id = s_ids[i * kMaxReqs + r];
            long long out = id;
            if (id >= 0 && a.d2t) {
                const int tgt = a.d2t[id];
                if (tgt < 0) atomicOr(a.status, kStatusIndex);
                out = tgt < 0 ? -1 : tgt;
            }
            a.out_ids[size_t(r) * a.k + i] = out;
        }
        if (nd == a.k && tid < a.B && ((live >> tid) & 1u)) a.prev[tid] = s_ids[(a.k - 1) * kMaxReqs + tid];
    }
    tc_fence_before();
    cluster_barrier();  // no CTA leaves while a store to it may be in flight
    tc_fence_after();
    if (warp == 0) tmem_dealloc(tmem, tmem_cols);
}

template <int NB, bool DBG>
dspark_status launch_cluster_nb(const CUtensorMap &tm2, const CUtensorMap &tm1, const CUtensorMap &tb,
                                const MarkovArgs &args, int R, int C, int nbuf, size_t smem, cudaStream_t stream) {
    auto kern = markov_cluster_kernel<NB, DBG>;
    static int configured_dev = -1;
    int dev = 0;
    cudaGetDevice(&dev);
    if (configured_dev != dev) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             static_cast<int>(kSmemLimit));
        if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute(markov_cluster smem)");
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
        if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute(markov_cluster cluster size)");
        configured_dev = dev;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(C));
    cfg.blockDim = dim3(kThreadsC);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = static_cast<unsigned>(C);
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t e = cudaLaunchKernelEx(&cfg, kern, tm2, tm1, tb, args, R, nbuf);
    if (e != cudaSuccess) return cuda_fail(e, "cudaLaunchKernelEx(markov_cluster)");
    return DSPARK_OK;
}

template <bool DBG>
dspark_status launch_cluster_dbg(const CUtensorMap &tm2, const CUtensorMap &tm1, const CUtensorMap &tb,
                                 const MarkovArgs &args, int R, int C, int nbuf, size_t smem, cudaStream_t stream) {
    if (args.B <= 1) return launch_cluster_nb<1, DBG>(tm2, tm1, tb, args, R, C, nbuf, smem, stream);
    if (args.B <= 2) return launch_cluster_nb<2, DBG>(tm2, tm1, tb, args, R, C, nbuf, smem, stream);
    if (args.B <= 4) return launch_cluster_nb<4, DBG>(tm2, tm1, tb, args, R, C, nbuf, smem, stream);
    return launch_cluster_nb<8, DBG>(tm2, tm1, tb, args, R, C, nbuf, smem, stream);
}

int nb_for(int B) { return B <= 1 ? 1 : B <= 2 ? 2 : B <= 4 ? 4 : 8; }

// Whether a cluster of 16 CTAs with the largest shared-memory request can be resident on
// the current device (cached per device).  Clusters of up to 8 always can.
bool cluster16_ok() {
    static int cached_dev = -1;
    static bool ok = false;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return false;
    if (cached_dev == dev) return ok;
    auto kern = markov_cluster_kernel<8, false>;
    ok = false;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(kSmemLimit)) ==
            cudaSuccess &&
        cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) == cudaSuccess) {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(16);
        cfg.blockDim = dim3(kThreadsC);
        cfg.dynamicSmemBytes = kSmemLimit;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = 16;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        int n = 0;
        ok = cudaOccupancyMaxActiveClusters(&n, kern, &cfg) == cudaSuccess && n >= 1;
    }
    cudaGetLastError();  // a refused query leaves no sticky error behind
    cached_dev = dev;
    return ok;
}

}  // namespace

int markov_cluster_size(int B, int V, int R, int k) {
    if (B < 1 || B > kMaxReqs || V < 4 || (V % 4) != 0 || k < 1 || (R != 64 && R != 128 && R != 256)) return 0;
    const int T = (V + kTileRowsC - 1) / kTileRowsC;
    const int cmax = cluster16_ok() ? 16 : 8;
    const int C = T < cmax ? T : cmax;
    const int ntile = (T + C - 1) / C;
    if (cluster_layout(ntile, R, nb_for(B), C, 1, k).total > kSmemLimit) return 0;
    return C;
}

dspark_status launch_markov_cluster(const MarkovArgs &args, int R, int C, cudaStream_t stream) {
    const int T = (args.V + kTileRowsC - 1) / kTileRowsC;
    if (C < 1 || C > kMaxCluster || C > T) return fail(DSPARK_ERR_INVALID, "markov_cluster: cluster size %d", C);
    const int ntile = (T + C - 1) / C;
    const int NB = nb_for(args.B);
    int nbuf = args.k < kMaxBaseBufs ? args.k : kMaxBaseBufs;
    while (nbuf > 1 && cluster_layout(ntile, R, NB, C, nbuf, args.k).total > kSmemLimit) --nbuf;
    const size_t smem = cluster_layout(ntile, R, NB, C, nbuf, args.k).total;
    if (smem > kSmemLimit) return fail(DSPARK_ERR_UNSUPPORTED, "markov_cluster: %zu bytes of shared memory", smem);
    CUtensorMap tm2, tm1, tb;
    const uint32_t nkb = static_cast<uint32_t>(R / 64);
    dspark_status st = make_tmap_kblocks(&tm2, args.w2, true, static_cast<uint64_t>(args.V), static_cast<uint64_t>(R),
                                         kTileRowsC, nkb);
    if (st != DSPARK_OK) return st;
    st = make_tmap_kblocks(&tm1, args.w1, true, static_cast<uint64_t>(args.V), static_cast<uint64_t>(R), kTileRowsC,
                           nkb);
    if (st != DSPARK_OK) return st;
    st = make_tmap_rows_f32(&tb, args.base, static_cast<uint64_t>(args.B), static_cast<uint64_t>(args.k),
                            static_cast<uint64_t>(args.V), static_cast<uint32_t>(args.B), kTileRowsC);
    if (st != DSPARK_OK) return st;
    if (args.dbg_logits || args.dbg_bias) return launch_cluster_dbg<true>(tm2, tm1, tb, args, R, C, nbuf, smem, stream);
    return launch_cluster_dbg<false>(tm2, tm1, tb, args, R, C, nbuf, smem, stream);
}

}  // namespace dspark
