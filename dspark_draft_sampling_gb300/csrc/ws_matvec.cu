// Weight-stationary small-M fp16 matvec: Y[M, N] = X[M, K] . W[N, K]^T on tcgen05.
//
// Method (SharpInference issue #441, sections "Observation", "Hypothesis" and "Proposed
// work"): the draft's fp16 projections have M = B = 7 rows; each weight element should be
// read from HBM once and applied to all M rows, so the kernel is bound by the weight
// stream.  On CUDA cores the multiply-adds, conversions and cross-lane sums cost about as
// many issue slots as the stream allows; here the contraction runs on the 5th-generation
// tensor cores, which leaves the SMs free to keep the stream going.
//
// GB300 design
//  * Work unit = (128 weight rows, a contiguous range of 64-wide k-blocks).  The split of K
//    per row block (S units) and the CTAs per SM (1 with a 10-stage ring, up to 3 with 4 stages)
//    are chosen per shape so that one wave of CTAs covers every unit with the smallest
//    largest load on any SM.
//  * Warp 4 (one thread) streams, per k-block, the W tile [128 rows x 64 k] (16 KB) and
//    the X tile [16 rows x 64 k] (2 KB; rows >= M read as zero) with 2-D TMA tensor copies
//    in the 128-byte-swizzled layout, through an mbarrier ring.  It initializes the barriers
//    and issues the first two stages before the CTA-wide set-up (TMEM allocation, the CTA
//    barrier), so the first tiles' DRAM latency overlaps that set-up.
//  * Warp 5 allocates 32 TMEM columns and one thread issues, per k-block, four
//    tcgen05.mma kind::f16 (M=128, N=16, K=16; fp16 in, fp32 accumulate) into TMEM.
//    tcgen05.commit frees each stage once its MMAs are done, and signals the epilogue
//    after the last one.
//  * Warps 0-3 (128 threads, one TMEM lane = one weight row each) load the 128 x 16
//    accumulator tile with tcgen05.ld.  With one unit per row block they write Y directly.
//    Otherwise the S units of a row block (S in {2, 4, 8}) are CTAs of one thread-block cluster
//    and reduce their fp32 partials in a fixed order, 0 + p_0 + p_1 + ... + p_{S-1}, so the
//    result is deterministic and does not depend on M: units 1..S-1 store their partial rows
//    into unit 0's shared memory (distributed shared memory), a cluster barrier, then unit 0
//    sums and writes Y.  A single-problem launch gives unit 0 a receive area of its own; a
//    grouped launch (several problems in one grid, clusters of the largest S, each problem's
//    units padded to whole clusters) reuses unit 0's ring once a first cluster barrier shows
//    every unit of the cluster done with its stream.  Both give the same bits, so a problem
//    gives the same result alone and in a group.
#include <cuda_fp16.h>

#include "tc.cuh"

namespace dspark {
namespace {

constexpr int kThreads = 192;      // warps 0-3 epilogue, 4 TMA, 5 MMA + TMEM
// Ring depth per launch: 10 x 18 KB stages with one CTA per SM; launches with more units than
// SMs take 4 stages in 74 KB, so three CTAs fit on an SM and each SM overlaps one CTA's fixed
// costs with the others' streams (measured on the grouped projections: one CTA per SM 53.0 us,
// two with 5 stages 47.1 us, three with 4 stages 43.0 us, the last in one wave; on a
// 151936 x 4096 matrix 187 / 184 / 180 us); fewer when a cluster's receive area needs the room.
constexpr int kStagesSolo = 10;
constexpr int kStagesShared = 4;
// Stages issued before the CTA barrier.  Issuing one stage (two TMA copies) takes the producing
// thread ~0.2 us, so a whole first ring issued there holds the MMAs back for microseconds;
// two are enough to cover the set-up (measured: single calls 0.4-0.8 us faster, others equal).
constexpr int kPreBarrierStages = 2;
constexpr int kMaxSplit = 8;       // units per row block (the portable cluster size)
constexpr int kRowsPerUnit = 128;  // MMA M
constexpr int kNPad = 16;          // MMA N: X rows padded to 16
constexpr int kKB = 64;            // k per block (128 bytes of fp16 = the swizzle span)
constexpr int kABytes = kRowsPerUnit * kKB * 2;  // 16 KB
constexpr int kBBytes = kNPad * kKB * 2;         // 2 KB
constexpr int kStageBytes = kABytes + kBBytes;   // 18 KB (multiple of 1024)
constexpr uint32_t kTmemCols = 32;
constexpr size_t kSmemSolo = 227 * 1024;         // per-CTA shared memory with one CTA per SM
constexpr size_t kSmemShared = 74 * 1024;        // ... with up to three
// dynamic shared memory: alignment slack, ring, cluster receive area, barriers and flags
constexpr size_t smem_bytes_for(int nst, size_t recv) { return 1024 + size_t(nst) * kStageBytes + recv + 256; }
// a grouped launch's unit 0 receives the other units' partial rows in its ring
static_assert(size_t(kStagesShared) * kStageBytes >= size_t(kMaxSplit - 1) * kRowsPerUnit * kNPad * 4,
              "the shared ring holds the partials of a split of kMaxSplit");
static_assert(smem_bytes_for(kStagesShared, 0) <= kSmemShared, "the shared ring fits its budget");

constexpr int kMaxProblems = 8;

struct WsProblem {
    void *Y;
    int y_fp32;
    int M, N, K;
    int nrb;    // row blocks (units beyond nrb * S are padding and stream nothing)
    int nkb;    // k-blocks
    int S;      // units per row block
    int unit0;  // first CTA of this problem in the grid (a multiple of the cluster size)
};

// Kernel parameters: up to P independent problems share one launch, CTA b taking unit
// b - unit0 of the problem whose range holds it.  The tensor maps stay in parameter space
// (__grid_constant__), where TMA reads them.  The scalars and problem descriptors come first:
// a CTA's first reads of the (cold) parameter block then fall on its first lines.  A
// single-problem launch uses P = 1, a parameter block of ~0.3 KB instead of ~2.5 KB.
template <int P>
struct WsGroupT {
    int nprob;
    int nst;            // ring stages
    int cluster;        // 0: no split problem; 1: one problem, unit 0 has a receive area;
                        // 2: grouped, unit 0's ring receives after a first cluster barrier
    int csize;          // cluster size (a multiple of every problem's S)
    int mcols;          // partial columns sent per row (8 or 16)
    unsigned *status;   // workspace status word: kWsStatusTimeout when a wait gave up
    unsigned long long timeout_ns;
    unsigned long long stall_ns;  // > 0 (fault-injection hook only): the epilogue first waits
                                  // this long on a barrier that nothing signals
    WsProblem prob[P];
    CUtensorMap tmW[P];
    CUtensorMap tmX[P];
};
using WsGroup = WsGroupT<kMaxProblems>;


// Address of the same shared-memory location in CTA `rank` of this cluster.
__device__ __forceinline__ uint32_t map_to_rank(uint32_t smem_addr_cta, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(smem_addr_cta), "r"(rank));
    return r;
}

__device__ __forceinline__ void st_cluster_v4(uint32_t addr, float a, float b, float c, float d) {
    asm volatile("st.shared::cluster.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "f"(a), "f"(b), "f"(c), "f"(d)
                 : "memory");
}

// Every thread of every CTA of the cluster; the warp must be converged (aligned form).
__device__ __forceinline__ void cluster_sync_all() {
    __syncwarp();
    asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
    asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

__device__ __forceinline__ void store_y(const WsProblem &a, int row, const float (&y)[kNPad]) {
#pragma unroll
    for (int m = 0; m < kNPad; ++m) {
        if (m < a.M) {
            const size_t o = size_t(m) * a.N + row;
            if (a.y_fp32)
                static_cast<float *>(a.Y)[o] = y[m];
            else
                static_cast<__half *>(a.Y)[o] = __float2half_rn(y[m]);
        }
    }
}

template <int P>
__global__ void __launch_bounds__(kThreads, 1) ws_matvec_tc_kernel(const __grid_constant__ WsGroupT<P> g) {
    extern __shared__ unsigned char smem_raw[];
    const uint32_t raw = smem_addr(smem_raw);
    unsigned char *smem = smem_raw + ((1024u - (raw & 1023u)) & 1023u);  // 1024-aligned tiles
    const int nst = g.nst;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    int pi = 0;
    while (pi + 1 < g.nprob && static_cast<int>(blockIdx.x) >= g.prob[pi + 1].unit0) ++pi;
    const WsProblem &a = g.prob[pi];
    const CUtensorMap *tmW = &g.tmW[pi];
    const CUtensorMap *tmX = &g.tmX[pi];
    const int unit = static_cast<int>(blockIdx.x) - a.unit0;
    const int rb = unit / a.S;
    const int sk = unit % a.S;
    // 32-bit: sk <= 8 and nkb < 2^25 (a 64-bit division would call a long out-of-line routine)
    const int kb0 = static_cast<int>(static_cast<unsigned>(sk) * static_cast<unsigned>(a.nkb) / static_cast<unsigned>(a.S));
    const int kb1 =
        static_cast<int>(static_cast<unsigned>(sk + 1) * static_cast<unsigned>(a.nkb) / static_cast<unsigned>(a.S));
    const int nk = rb < a.nrb ? kb1 - kb0 : 0;  // padding units stream nothing
    const int n0 = rb * kRowsPerUnit;
    // split row blocks: unit 0 of the row block receives the other units' partial rows,
    // [S - 1][128 rows][mcols] fp32, in its own area (cluster mode 1) or its ring (mode 2)
    const size_t recv_bytes = g.cluster == 1 ? size_t(a.S - 1) * kRowsPerUnit * g.mcols * 4 : 0;
    float *recv = reinterpret_cast<float *>(smem + (g.cluster == 1 ? size_t(nst) * kStageBytes : 0));
    const uint32_t leader =
        static_cast<uint32_t>(static_cast<int>(blockIdx.x) % g.csize - sk);  // cluster rank of unit 0
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + size_t(nst) * kStageBytes + recv_bytes);
    uint64_t *empty = full + nst;
    uint64_t *done = empty + nst;
    uint64_t *never = done + 1;  // signalled by nobody: the fault-injection hook waits on it
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(never + 1);

    if (warp == 4 && lane == 0) {
        // The producer sets up the barriers and starts the first copies before the CTA-wide
        // set-up, so the DRAM latency of the first tiles overlaps it.
        for (int s = 0; s < nst; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        mbar_init(done, 1);
        mbar_init(never, 1);
        fence_mbar_init();
        pdl_wait();  // no global-memory access before this point
        const uint64_t pol_w = l2_policy_evict_first();
        const uint64_t pol_x = l2_policy_evict_last();
        for (int j = 0; j < nk && j < nst && j < kPreBarrierStages; ++j) {
            unsigned char *sa = smem + size_t(j) * kStageBytes;
            mbar_arrive_expect_tx(&full[j], kStageBytes);
            tma_load_2d(sa, tmW, (kb0 + j) * kKB, n0, &full[j], pol_w);
            tma_load_2d(sa + kABytes, tmX, (kb0 + j) * kKB, 0, &full[j], pol_x);
        }
    }
    if (warp == 5) tmem_alloc(tmem_slot, kTmemCols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    pdl_launch_dependents();
    pdl_wait();  // no global-memory access before this point

    if (warp == 4) {
        // ---- TMA producer: the copies after the first ones ----
        if (lane == 0) {
            const uint64_t pol_w = l2_policy_evict_first();
            const uint64_t pol_x = l2_policy_evict_last();
            // k-block j uses slot j % nst; from the second pass on, the slot must first be
            // freed by the MMAs of k-block j - nst
            const int first = nst < kPreBarrierStages ? nst : kPreBarrierStages;
            for (int j = first; j < nk; ++j) {
                const int st = j % nst;
                if (j >= nst && !mbar_wait(&empty[st], static_cast<uint32_t>(((j / nst) & 1) ^ 1), g.timeout_ns)) {
                    atomicOr(g.status, kWsStatusTimeout);
                    break;
                }
                unsigned char *sa = smem + size_t(st) * kStageBytes;
                mbar_arrive_expect_tx(&full[st], kStageBytes);
                tma_load_2d(sa, tmW, (kb0 + j) * kKB, n0, &full[st], pol_w);
                tma_load_2d(sa + kABytes, tmX, (kb0 + j) * kKB, 0, &full[st], pol_x);
            }
        }
    } else if (warp == 5) {
        // ---- MMA issuer ----
        if (lane == 0) {
            constexpr uint32_t idesc = idesc_f16(false, kRowsPerUnit, kNPad);
            // descriptors built once, advanced by byte offsets >> 4 (shared memory < 256 KB)
            const uint64_t dA0 = smem_desc_sw128(smem_addr(smem));
            int st = 0;
            uint32_t ph = 0;
            for (int j = 0; j < nk; ++j) {
                if (!mbar_wait(&full[st], ph, g.timeout_ns)) {
                    atomicOr(g.status, kWsStatusTimeout);
                    break;
                }
                tc_fence_after();
                const uint64_t dA = dA0 + static_cast<uint64_t>(st * (kStageBytes >> 4));
                const uint64_t dB = dA + static_cast<uint64_t>(kABytes >> 4);
                tc_mma_f16(tmem, dA, dB, idesc, j != 0);  // K = 16 per MMA, 32 B apart
                tc_mma_f16(tmem, dA + 2, dB + 2, idesc, 1u);
                tc_mma_f16(tmem, dA + 4, dB + 4, idesc, 1u);
                tc_mma_f16(tmem, dA + 6, dB + 6, idesc, 1u);
                tc_commit(&empty[st]);
                if (++st == nst) {
                    st = 0;
                    ph ^= 1u;
                }
            }
            tc_commit(done);
        }
    } else {
        // ---- epilogue: warp w owns TMEM lanes / weight rows 32w .. 32w+31 ----
        if (g.stall_ns && !mbar_wait(never, 0, g.stall_ns) && threadIdx.x == 0) atomicOr(g.status, kWsStatusTimeout);
        const bool ok = mbar_wait(done, 0, g.timeout_ns);
        if (!ok) atomicOr(g.status, kWsStatusTimeout);
        tc_fence_after();
        uint32_t v[16];
        tmem_ld_16(tmem + (static_cast<uint32_t>(warp * 32) << 16), v);
        const int lrow = warp * 32 + lane;
        const int row = n0 + lrow;
        if (a.S == 1) {
            if (ok && row < a.N) {
                float y[kNPad];
#pragma unroll
                for (int m = 0; m < kNPad; ++m) y[m] = __uint_as_float(v[m]);
                store_y(a, row, y);
            }
        } else {
            // units 1..S-1: this row's partial goes into unit 0's receive area; in a grouped
            // launch that is unit 0's ring, idle once every unit of the cluster has passed the
            // first barrier (every unit's stream is done by then)
            if (g.cluster == 2) cluster_sync_all();
            if (sk != 0) {
                const uint32_t dst = map_to_rank(
                    smem_addr(recv + (size_t(sk - 1) * kRowsPerUnit + lrow) * g.mcols), leader);
#pragma unroll
                for (int q = 0; q < kNPad / 4; ++q)
                    if (4 * q < g.mcols)
                        st_cluster_v4(dst + 16u * q, __uint_as_float(v[4 * q]), __uint_as_float(v[4 * q + 1]),
                                      __uint_as_float(v[4 * q + 2]), __uint_as_float(v[4 * q + 3]));
            }
            cluster_sync_all();  // orders the stores before unit 0 reads them
            if (sk == 0 && ok && row < a.N) {
                // y[m] = 0 + p_0[m] + p_1[m] + ... + p_{S-1}[m]
                float y[kNPad];
#pragma unroll
                for (int m = 0; m < kNPad; ++m) y[m] = 0.f + __uint_as_float(v[m]);
                for (int s = 1; s < a.S; ++s) {
                    const float4 *src = reinterpret_cast<const float4 *>(recv + (size_t(s - 1) * kRowsPerUnit + lrow) * g.mcols);
#pragma unroll
                    for (int q = 0; q < kNPad / 4; ++q) {
                        if (4 * q < g.mcols) {
                            const float4 t = src[q];
                            y[4 * q] += t.x;
                            y[4 * q + 1] += t.y;
                            y[4 * q + 2] += t.z;
                            y[4 * q + 3] += t.w;
                        }
                    }
                }
                store_y(a, row, y);
            }
        }
    }
    // split row blocks: every other thread of the CTA takes part in the cluster barriers
    if (a.S > 1 && warp >= 4) {
        if (g.cluster == 2) cluster_sync_all();
        cluster_sync_all();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 5) tmem_dealloc(tmem, kTmemCols);
}

struct Plan {
    int nrb, nkb, S;
    int cps;  // 1: split sized for one CTA per SM; 2: the shared ring, several CTAs per SM
};

// Receive area of a cluster launch: (S - 1) partial tiles of 128 rows x mcols fp32.
size_t recv_bytes_for(int S, int M) { return size_t(S - 1) * kRowsPerUnit * (M <= 8 ? 8 : 16) * 4; }

// Ring stages that fit with `cps` CTAs per SM next to a receive area of `recv` bytes.
int stages_for(int cps, size_t recv) {
    const size_t budget = cps == 1 ? kSmemSolo : kSmemShared;
    const int cap = cps == 1 ? kStagesSolo : kStagesShared;
    const long long fit = (static_cast<long long>(budget) - static_cast<long long>(smem_bytes_for(0, recv))) / kStageBytes;
    return static_cast<int>(fit < cap ? fit : cap);
}

// Whether one wave of a cluster launch holds `units` CTAs in clusters of S (cached per device
// and shape of the question).
bool clusters_fit(int S, int cps, int M, int units);

// The split of K: for S in {1, 2, 4, 8} units per row block with one CTA per SM, the largest
// number of k-blocks any SM streams when every unit is resident in one wave; the smallest wins,
// then the smaller S.  A shape with more row blocks than SMs runs unsplit with the shared ring
// (up to three CTAs per SM).  (Splits sized for two CTAs per SM were measured about 1 us faster
// alone on the 12288-row and 12288-wide projections, but their extra short units slowed the
// grouped launch of the four projections, so they are not used.)  S is a power of two so that
// one cluster size serves every problem of a grouped launch.  Whether the clusters fit is
// asked for the largest receive area (M = 16), so the split depends on N and K only and a
// problem is split the same way in a single and in a grouped launch.
Plan plan_for(int N, int K, int sms) {
    Plan p;
    p.nrb = (N + kRowsPerUnit - 1) / kRowsPerUnit;
    p.nkb = (K + kKB - 1) / kKB;
    p.S = 1;
    p.cps = 2;
    long long best = -1;
    for (int S = 1; S <= kMaxSplit && S <= p.nkb; S *= 2) {
        const long long units = static_cast<long long>(p.nrb) * S;
        if (units > sms) break;
        if (stages_for(1, recv_bytes_for(S, 16)) < 3) break;
        if (S > 1 && !clusters_fit(S, 1, 16, static_cast<int>(units))) continue;
        const long long load = (p.nkb + S - 1) / S;  // one CTA per SM: its k-blocks
        if (best < 0 || load < best) {
            best = load;
            p.S = S;
            p.cps = 1;
        }
    }
    return p;
}

// ---- cluster occupancy, queried once per device and (S, cps, receive size) ----------------
dspark_status configure_kernel(int dev) {
    static int configured_dev = -1;
    if (configured_dev == dev) return DSPARK_OK;
    const void *kerns[2] = {reinterpret_cast<const void *>(ws_matvec_tc_kernel<1>),
                            reinterpret_cast<const void *>(ws_matvec_tc_kernel<kMaxProblems>)};
    for (const void *kern : kerns) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             static_cast<int>(kSmemSolo));
        if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute(ws_matvec)");
        int per_sm = 0;
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kThreads, smem_bytes_for(kStagesSolo, 0));
        if (e != cudaSuccess) return cuda_fail(e, "cudaOccupancyMaxActiveBlocksPerMultiprocessor(ws_matvec)");
        if (per_sm < 1) return fail(DSPARK_ERR_CUDA, "ws_matvec kernel cannot be resident on an SM");
    }
    configured_dev = dev;
    return DSPARK_OK;
}

bool clusters_fit(int S, int cps, int M, int units) {
    struct Entry {
        int dev, S, cps, mc, clusters;
    };
    static Entry cache[64];
    static int n = 0;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return false;
    const int mc = M <= 8 ? 8 : 16;
    int clusters = -1;
    for (int i = 0; i < n; ++i)
        if (cache[i].dev == dev && cache[i].S == S && cache[i].cps == cps && cache[i].mc == mc) clusters = cache[i].clusters;
    if (clusters < 0) {
        if (configure_kernel(dev) != DSPARK_OK) return false;
        const size_t recv = recv_bytes_for(S, M);
        const int nst = stages_for(cps, recv);
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(static_cast<unsigned>(S));
        cfg.blockDim = dim3(kThreads);
        cfg.dynamicSmemBytes = smem_bytes_for(nst, recv);
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = static_cast<unsigned>(S);
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        int c = 0;
        if (cudaOccupancyMaxActiveClusters(&c, ws_matvec_tc_kernel<1>, &cfg) != cudaSuccess) {
            cudaGetLastError();
            c = 0;
        }
        clusters = c;
        if (n < 64) cache[n++] = Entry{dev, S, cps, mc, clusters};
    }
    return static_cast<long long>(clusters) * S >= units;
}

}  // namespace
}  // namespace dspark

extern "C" size_t dspark_ws_matvec_workspace_bytes(int M, int N, int K) {
    // split rows reduce in distributed shared memory: the workspace holds the status word
    (void)M;
    (void)N;
    (void)K;
    return dspark::kWsHeaderBytes;
}

namespace {

// Checks one problem; returns DSPARK_OK with *skip set when it has nothing to do.
dspark_status check_problem(const dspark_ws_problem &q, bool *skip) {
    using namespace dspark;
    *skip = false;
    if (q.M < 0 || q.N < 0 || q.K < 0) return fail(DSPARK_ERR_INVALID, "ws_matvec: negative size");
    if (q.M > 16) return fail(DSPARK_ERR_UNSUPPORTED, "ws_matvec: M=%d > 16", q.M);
    if (q.K < 8 || (q.K % 8) != 0) return fail(DSPARK_ERR_INVALID, "ws_matvec: K=%d must be a positive multiple of 8", q.K);
    if (q.M == 0 || q.N == 0) {
        *skip = true;
        return DSPARK_OK;
    }
    if (!q.W || !q.X || !q.Y) return fail(DSPARK_ERR_INVALID, "ws_matvec: null pointer argument");
    if (!aligned(q.W, 16) || !aligned(q.X, 16)) return fail(DSPARK_ERR_INVALID, "ws_matvec: W and X must be 16-byte aligned");
    if (!aligned(q.Y, q.y_is_fp32 ? 4 : 2)) return fail(DSPARK_ERR_INVALID, "ws_matvec: misaligned Y");
    return DSPARK_OK;
}

// Workspace of a group: the status word (split rows reduce in distributed shared memory).
size_t group_workspace_bytes(const dspark_ws_problem *probs, int n, int sms) {
    (void)probs;
    (void)n;
    (void)sms;
    return dspark::kWsHeaderBytes;
}

dspark_status ws_enqueue_group(const dspark_ws_problem *probs, int n, void *workspace, size_t workspace_bytes,
                               unsigned long long stall_ns, dspark_stream_t stream) {
    using namespace dspark;
    clear_error();
    if (n < 0 || n > kMaxProblems) return fail(DSPARK_ERR_UNSUPPORTED, "ws_matvec: %d problems (at most %d)", n, kMaxProblems);
    if (n > 0 && !probs) return fail(DSPARK_ERR_INVALID, "ws_matvec: null problem array");
    int live = 0;
    for (int i = 0; i < n; ++i) {
        bool skip = false;
        const dspark_status st = check_problem(probs[i], &skip);
        if (st != DSPARK_OK) return st;
        live += skip ? 0 : 1;
    }
    if (live == 0) return DSPARK_OK;  // nothing to enqueue
    if (!workspace) return fail(DSPARK_ERR_INVALID, "ws_matvec: null workspace");
    if (!aligned(workspace, 256)) return fail(DSPARK_ERR_INVALID, "ws_matvec: workspace must be 256-byte aligned");
    int sms = 0;
    int rc = current_sm_count(&sms);
    if (rc != DSPARK_OK) return static_cast<dspark_status>(rc);
    const size_t need = group_workspace_bytes(probs, n, sms);
    if (workspace_bytes < need)
        return fail(DSPARK_ERR_INVALID, "ws_matvec: workspace of %zu bytes < required %zu", workspace_bytes, need);
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    dspark_status st = configure_kernel(dev);
    if (st != DSPARK_OK) return st;

    WsGroup g;
    g.nprob = 0;
    g.status = static_cast<unsigned *>(workspace);
    g.timeout_ns = kDefaultTimeoutNs;
    g.stall_ns = stall_ns;
    // The grid takes the problems with the longest units first (longest-processing-time
    // order), so the last wave holds short units and the tail stays short.  The order changes
    // no result: every problem keeps its own split and summation order.
    int order[kMaxProblems];
    Plan plans[kMaxProblems];
    int norder = 0;
    for (int i = 0; i < n; ++i)
        if (probs[i].M != 0 && probs[i].N != 0) {
            plans[norder] = plan_for(probs[i].N, probs[i].K, sms);
            order[norder++] = i;
        }
    auto unit_blocks = [&](int j) { return (plans[j].nkb + plans[j].S - 1) / plans[j].S; };
    int idx[kMaxProblems];
    for (int j = 0; j < norder; ++j) idx[j] = j;
    for (int a = 1; a < norder; ++a)  // stable insertion sort, longest units first
        for (int b = a; b > 0 && unit_blocks(idx[b]) > unit_blocks(idx[b - 1]); --b) {
            const int t = idx[b];
            idx[b] = idx[b - 1];
            idx[b - 1] = t;
        }
    // cluster size: the largest split (every split is a power of two, so it divides this one)
    int csize = 1, mmax = 0;
    for (int j = 0; j < norder; ++j) {
        csize = plans[j].S > csize ? plans[j].S : csize;
        mmax = probs[order[j]].M > mmax ? probs[order[j]].M : mmax;
    }
    g.csize = csize;
    g.mcols = mmax <= 8 ? 8 : 16;
    g.cluster = csize == 1 ? 0 : (live == 1 ? 1 : 2);
    unsigned units = 0;
    for (int oj = 0; oj < norder; ++oj) {
        const int jj = idx[oj];
        const dspark_ws_problem &q = probs[order[jj]];
        const Plan &p = plans[jj];
        const int j = g.nprob++;
        st = make_tmap_2d(&g.tmW[j], q.W, false, static_cast<uint64_t>(q.N), static_cast<uint64_t>(q.K), kRowsPerUnit,
                          kKB);
        if (st != DSPARK_OK) return st;
        st = make_tmap_2d(&g.tmX[j], q.X, false, static_cast<uint64_t>(q.M), static_cast<uint64_t>(q.K), kNPad, kKB);
        if (st != DSPARK_OK) return st;
        WsProblem &a = g.prob[j];
        a.Y = q.Y;
        a.y_fp32 = q.y_is_fp32 ? 1 : 0;
        a.M = q.M;
        a.N = q.N;
        a.K = q.K;
        a.nrb = p.nrb;
        a.nkb = p.nkb;
        a.S = p.S;
        a.unit0 = static_cast<int>(units);
        // whole clusters per problem: the last one may hold padding units
        const unsigned pu = static_cast<unsigned>(p.nrb) * static_cast<unsigned>(p.S);
        units += (pu + static_cast<unsigned>(csize) - 1) / static_cast<unsigned>(csize) * static_cast<unsigned>(csize);
    }

    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    size_t recv = 0;
    if (live == 1) {
        // one problem: the ring sized for the CTAs per SM its split assumed, and for S > 1 a
        // receive area for unit 0
        recv = csize > 1 ? recv_bytes_for(csize, g.prob[0].M) : 0;
        g.nst = stages_for(plans[0].cps, recv);
    } else {
        // more units than SMs: the shallower ring, up to three CTAs per SM (unit 0 receives
        // the partials in its ring, whose 72 KB hold (S - 1) x 128 x 16 fp32 even at S = 8)
        g.nst = units > static_cast<unsigned>(sms) ? kStagesShared : kStagesSolo;
    }
    if (csize > 1) {
        attr[1].id = cudaLaunchAttributeClusterDimension;
        attr[1].val.clusterDim.x = static_cast<unsigned>(csize);
        attr[1].val.clusterDim.y = 1;
        attr[1].val.clusterDim.z = 1;
        cfg.numAttrs = 2;
    }
    cfg.gridDim = dim3(units);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem_bytes_for(g.nst, recv);
    cfg.stream = reinterpret_cast<cudaStream_t>(stream);
    if (g.nprob == 1) {  // the small parameter block
        WsGroupT<1> g1;
        g1.nprob = 1;
        g1.nst = g.nst;
        g1.cluster = g.cluster;
        g1.csize = g.csize;
        g1.mcols = g.mcols;
        g1.status = g.status;
        g1.timeout_ns = g.timeout_ns;
        g1.stall_ns = g.stall_ns;
        g1.prob[0] = g.prob[0];
        g1.tmW[0] = g.tmW[0];
        g1.tmX[0] = g.tmX[0];
        e = cudaLaunchKernelEx(&cfg, ws_matvec_tc_kernel<1>, g1);
    } else {
        e = cudaLaunchKernelEx(&cfg, ws_matvec_tc_kernel<kMaxProblems>, g);
    }
    if (e != cudaSuccess) return cuda_fail(e, "ws_matvec launch");
    return DSPARK_OK;
}

dspark_status ws_enqueue(const uint16_t *W, const uint16_t *X, void *Y, int y_is_fp32, int M, int N, int K,
                         void *workspace, size_t workspace_bytes, unsigned long long stall_ns, dspark_stream_t stream) {
    const dspark_ws_problem q = {W, X, Y, y_is_fp32, M, N, K};
    return ws_enqueue_group(&q, 1, workspace, workspace_bytes, stall_ns, stream);
}

}  // namespace

extern "C" dspark_status dspark_ws_matvec(const uint16_t *W, const uint16_t *X, void *Y, int y_is_fp32, int M, int N,
                                          int K, void *workspace, size_t workspace_bytes, dspark_stream_t stream) {
    return ws_enqueue(W, X, Y, y_is_fp32, M, N, K, workspace, workspace_bytes, 0ull, stream);
}

extern "C" size_t dspark_ws_matvec_grouped_workspace_bytes(const dspark_ws_problem *problems, int n_problems) {
    if (n_problems < 0 || (n_problems > 0 && !problems)) return 0;
    int sms = 0;
    if (dspark::current_sm_count(&sms) != DSPARK_OK) return 0;
    return group_workspace_bytes(problems, n_problems, sms);
}

extern "C" dspark_status dspark_ws_matvec_grouped(const dspark_ws_problem *problems, int n_problems, void *workspace,
                                                  size_t workspace_bytes, dspark_stream_t stream) {
    return ws_enqueue_group(problems, n_problems, workspace, workspace_bytes, 0ull, stream);
}

extern "C" dspark_status dspark_ws_matvec_debug(const uint16_t *W, const uint16_t *X, void *Y, int y_is_fp32, int M,
                                                int N, int K, void *workspace, size_t workspace_bytes,
                                                unsigned stall_us, dspark_stream_t stream) {
    if (stall_us == 0) return dspark::fail(DSPARK_ERR_INVALID, "ws_matvec_debug: stall_us must be > 0");
    return ws_enqueue(W, X, Y, y_is_fp32, M, N, K, workspace, workspace_bytes, 1000ull * stall_us, stream);
}

extern "C" dspark_status dspark_ws_matvec_status(void *workspace, dspark_stream_t stream) {
    using namespace dspark;
    clear_error();
    if (!workspace) return fail(DSPARK_ERR_INVALID, "ws_matvec_status: null workspace");
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    cudaError_t e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
    unsigned st = 0;
    e = cudaMemcpy(&st, workspace, sizeof st, cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return cuda_fail(e, "cudaMemcpy(ws status)");
    if (st == 0) return DSPARK_OK;
    // report once, and leave the workspace zero-filled again
    e = cudaMemset(workspace, 0, sizeof st);
    if (e != cudaSuccess) return cuda_fail(e, "cudaMemset(ws status)");
    return fail(DSPARK_ERR_TIMEOUT, "ws_matvec: a device-side wait timed out");
}
