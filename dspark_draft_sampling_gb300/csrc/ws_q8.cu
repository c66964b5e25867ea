// Weight-stationary small-M matvec with Q8_0 weights: Y[M, N] = X[M, K] . dequant(W)[N, K]^T.
//
// Method (SharpInference issue #441, "Proposed work"): the weight-stationary kernels of its
// #194 read quantized weights, streaming each weight once for all M rows; the issue notes
// that an SoA repack may be needed.  Weights here are Q8_0 (per 32 elements of a row: an
// fp16 scale d and 32 int8 q; weight = d * q).
//
// Layout: dspark_q8_0_repack turns the ggml array of 34-byte blocks into two row-major
// arrays, q int8 [N, K] and d fp16 [N, K/32], so the int8 tiles can be moved by 2-D TMA
// tensor copies (the 34-byte blocks cannot).
//
// Arithmetic: the dequantized weight d * q has up to 18 significant bits, so it cannot be a
// 16-bit tensor-core operand without rounding; q itself can (every int8 is an fp16 number).
// The kernel therefore runs one tcgen05 MMA group per Q8_0 block:
//     S[n, b, m] = sum_{j<32} q[n, 32b + j] * X[m, 32b + j]     (fp16 x fp16 products, exact;
//                                                                 fp32 accumulation in TMEM)
// and the epilogue applies the scale in fp32:  y[n, m] += d[n, b] * S[n, b, m], blocks in k
// order.  Every output is summed in one fixed order (blocks, then split-K units in order), so
// results are deterministic and row m's does not depend on M.
//
// GB300 design (one CTA per SM, 15 warps)
//  * Work unit = (128 weight rows, a range of 256-k superblocks).  With at most as many row
//    blocks as SMs, K is split into S <= 8 units per row block, one unit per CTA, S chosen for
//    the fewest superblocks per CTA in one wave, and the S CTAs of a row block form a
//    thread-block cluster.  With more row blocks than SMs the CTAs are persistent: each takes
//    every gridDim.x-th unit and streams the stages of its units back to back, so one unit's
//    epilogue overlaps the next unit's loads.
//  * Warp 12 (one thread) streams, per 128-k stage, the int8 tile [128 rows x 128 k] (16 KB,
//    128-byte swizzle, one 3-D copy of a single 128-byte column atom) and the X tile [16 rows x 128 k] (two 2 KB fp16 atoms in one 3-D copy;
//    rows >= M read as zero) with TMA tensor copies through a 10-stage ring (200 KB).
//  * Warps 4-7 take the even stages and warps 8-11 the odd ones: each thread converts one weight
//    row's 128 int8 to fp16 (a byte permute puts q + 128 into the mantissa of 1024, one packed
//    subtraction of 1152 leaves q exactly) and writes them with tcgen05.st straight into tensor
//    memory, where the MMA takes its A operand: the fp16 copy never touches shared memory.
//  * Warp 13 allocates all 512 TMEM columns (16 accumulator slots of 128 x 16 fp32 and a 4-slot
//    ring of fp16 A tiles).  Warps 13 and 14 issue the MMAs of the even and odd stages: per
//    Q8_0 block two tcgen05.mma kind::f16 (M=128, N=16, K=16; A from TMEM, B = X from shared
//    memory) into a fresh accumulator slot, and one tcgen05.commit per stage, which hands the
//    stage's 4 slots to the epilogue and frees its A tile and its shared-memory slot.  A
//    single issuing thread spends far longer per MMA than the tensor pipe does (the barrier
//    waits and the commit of each stage, slowed further while the converters stream
//    tcgen05.st), and issuers in separate warps proceed in parallel.  The issuer count must
//    divide the 4 A slots / accumulator groups: each issuer then also handled the previous
//    use of every slot it waits on (stage J - 4), so the slot's barriers are never more than
//    one phase from the one it waits for and the parity wait is exact.  With three issuers
//    stage J - 4 belongs to another issuer, a lagging converter leaves the barrier a whole
//    phase behind, the parity test passes early and the MMAs read a half-written A tile.
//  * Warps 0-3 (one TMEM lane = one weight row per thread) read a stage's 4 x 16 sums with
//    tcgen05.ld and fold them in with the row's scales (loaded 8 at a time from global memory,
//    four loads ahead).
//    With one unit per row block they write Y directly.  Otherwise, after a cluster barrier
//    (every unit of the row block has finished streaming, so unit 0's ring is idle), units
//    1..S-1 store their partial rows into unit 0's ring through distributed shared memory and,
//    after a second barrier, unit 0 sums 0 + p_0 + p_1 + ... + p_{S-1} and writes Y.
#include <cuda_fp16.h>

#include "tc.cuh"

namespace dspark {
namespace {

constexpr int kConvWarps = 8;          // two groups of 4, alternate stages
constexpr int kTmaWarp = 4 + kConvWarps;
constexpr int kMmaWarp = kTmaWarp + 1;  // first of kMmaIssuers warps
constexpr int kMmaIssuers = 2;         // issuer i takes the stages J = i mod 2
constexpr int kThreads = 32 * (kMmaWarp + kMmaIssuers);  // 480: warps 0-3 epilogue, 4-11 convert, 12 TMA, 13-14 MMA
constexpr int kRows = 128;             // weight rows per unit: MMA M, TMEM lanes
constexpr int kNPad = 16;              // MMA N: X rows padded to 16
constexpr int kKS = 128;               // k per stage: 128 B of int8 per row (the 128-byte swizzle span)
constexpr int kBlocksPerStage = kKS / 32;   // 4 Q8_0 blocks
constexpr int kSuper = 2;              // stages per 256-k superblock (8 scales of a row)
constexpr int kStages = 10;            // shared-memory ring (even, so each stage parity keeps its slots)
constexpr int kPreBarrierStages = 2;   // stages issued before the CTA-wide set-up
constexpr int kMaxSplit = 8;           // units per row block (the portable cluster size)
constexpr int kQBytes = kRows * kKS;                // 16 KB int8 tile
constexpr int kXAtomBytes = kNPad * 64 * 2;         // 2 KB: 16 rows x 64 fp16
constexpr int kSlotBytes = kQBytes + 2 * kXAtomBytes;  // 20 KB (multiple of 1024)
constexpr int kTSlots = 16;            // TMEM accumulator slots (4 stages x 4 blocks)
constexpr int kTGroups = kTSlots / kBlocksPerStage;  // one group per stage
constexpr int kASlots = 4;             // TMEM ring of fp16 A tiles
constexpr uint32_t kACols = kKS / 2;   // 64 columns: 128 fp16 per lane
constexpr uint32_t kAColBase = kTSlots * kNPad;                  // 256
constexpr uint32_t kTmemCols = kAColBase + kASlots * kACols;     // 512
constexpr int kNumBars = 2 * kStages + kASlots + kTGroups + kMmaIssuers + 1;
constexpr size_t kSmemBytes = 1024 + size_t(kStages) * kSlotBytes + kNumBars * 8 + 16;
static_assert(kTmemCols == 512, "the TMEM allocation must be a power of two <= 512");
static_assert(kStages % 2 == 0 && kASlots % 2 == 0 && kTGroups % 2 == 0, "rings must keep stage parity");
static_assert(kASlots == kTGroups && kASlots < kStages, "stage j uses A slot and accumulator group j % 4");
static_assert(kASlots % kMmaIssuers == 0 && kASlots % 2 == 0,
              "the issuer (and the converter group) of stage j must also own stage j - kASlots, "
              "so that its parity waits on the slot's barriers are exact");

constexpr int kMaxProblems = 8;

struct Q8Problem {
    const uint16_t *d;  // [N, K/32] fp16 scales
    void *Y;
    int y_fp32;
    int M, N, K;
    int nsb;    // 256-k superblocks
    int S;      // units per row block
    int nrb;    // row blocks (units beyond nrb * S are padding and stream nothing)
    int unit0;  // first unit of the problem (a multiple of the cluster size)
    int mcols;  // cluster mode: partial columns sent per row (8 or 16)
    int sb_base;  // stream-K mode: the problem's first superblock in the launch's sequence
};

// Kernel parameters: up to P problems share one launch.  Units are numbered across the
// problems, problem p holding units unit0 .. (next problem's unit0) - 1; CTA c takes units c,
// c + gridDim.x, ...  The tensor maps stay in parameter space (__grid_constant__), where TMA
// reads them.  A single-problem launch uses P = 1.
template <int P>
struct Q8GroupT {
    int nprob;
    int units;
    int cluster;  // 1: one unit per CTA, and the S units of a row block are CTAs of one cluster
    int csize;    // cluster size (a multiple of every problem's S; 1 without clusters)
    unsigned *status;   // workspace status word: kWsStatusTimeout when a wait gave up
    unsigned long long timeout_ns;
    unsigned long long stall_ns;  // > 0 (fault-injection hook only): the epilogue first waits
                                  // this long on a barrier that nothing signals
    Q8Problem prob[P];
    CUtensorMap tmQ[P];
    CUtensorMap tmX[P];
    // Stream-K mode (grouped launches): the row blocks of all problems, each K-long, form one
    // sequence of total_sb superblocks; CTA c takes superblocks [c T / G, (c + 1) T / G).  A
    // row block split between CTAs is finished by the CTA holding its first superblocks, which
    // adds the later CTAs' partial rows (partials[c], flags[c]) in CTA order.
    int streamk;
    int total_sb;
    float *partials;   // [grid][128][16] fp32
    unsigned *flags;   // [grid]: 1 while partials[c] holds a row block's later part
    int withheld_flag;  // fault-injection hook only (else -1): this CTA writes its partial but
                        // never sets its flag, so the CTA finishing that row block gives up
};

struct Unit {
    int p, rb, sk, sb0, nsup, nst, ks0, n0;
};

// First superblock of CTA c's range in stream-K mode.
__device__ __forceinline__ int range_begin(int c, int total_sb, int G) {
    return static_cast<int>(static_cast<long long>(c) * total_sb / G);
}

// The CTA's work in order: its units c, c + gridDim.x, ..., or in stream-K mode the pieces of
// row blocks its superblock range covers.
struct Cursor {
    int u;         // unit mode: the next unit
    int gsb, end;  // stream-K mode: the next superblock and the end of the range
};

template <int P>
__device__ __forceinline__ Unit unit_geometry(const Q8GroupT<P> &grp, int u) {
    Unit g;
    int p = 0;
    while (p + 1 < grp.nprob && u >= grp.prob[p + 1].unit0) ++p;
    const Q8Problem &a = grp.prob[p];
    const int v = u - a.unit0;
    g.p = p;
    g.rb = v / a.S;
    g.sk = v % a.S;
    // 32-bit: sk <= 8 and nsb < 2^23
    g.sb0 = static_cast<int>(static_cast<unsigned>(g.sk) * static_cast<unsigned>(a.nsb) / static_cast<unsigned>(a.S));
    const int sb1 =
        static_cast<int>(static_cast<unsigned>(g.sk + 1) * static_cast<unsigned>(a.nsb) / static_cast<unsigned>(a.S));
    g.nsup = g.rb < a.nrb ? sb1 - g.sb0 : 0;  // padding units stream nothing
    g.nst = g.nsup * kSuper;   // 128-k stages
    g.ks0 = g.sb0 * kSuper;    // first 128-k stage index along K
    g.n0 = g.rb * kRows;
    return g;
}

template <bool SK, int P>
__device__ __forceinline__ Cursor cursor_begin(const Q8GroupT<P> &g) {
    Cursor c;
    c.u = blockIdx.x;
    c.gsb = 0;
    c.end = 0;
    if constexpr (SK) {
        c.gsb = range_begin(blockIdx.x, g.total_sb, gridDim.x);
        c.end = range_begin(blockIdx.x + 1, g.total_sb, gridDim.x);
    }
    return c;
}

template <bool SK, int P>
__device__ __forceinline__ bool cursor_next(const Q8GroupT<P> &g, Cursor &c, Unit &out) {
    if constexpr (!SK) {
        if (c.u >= g.units) return false;
        out = unit_geometry(g, c.u);
        c.u += gridDim.x;
        return true;
    }
    if (c.gsb >= c.end) return false;
    int p = 0;
    while (p + 1 < g.nprob && c.gsb >= g.prob[p + 1].sb_base) ++p;
    const Q8Problem &a = g.prob[p];
    const int off = c.gsb - a.sb_base;
    out.p = p;
    out.rb = off / a.nsb;
    out.sk = 0;
    out.sb0 = off - out.rb * a.nsb;
    const int left = a.nsb - out.sb0;
    out.nsup = left < c.end - c.gsb ? left : c.end - c.gsb;
    out.nst = out.nsup * kSuper;
    out.ks0 = out.sb0 * kSuper;
    out.n0 = out.rb * kRows;
    c.gsb += out.nsup;
    return true;
}

// Two int8 values (bytes of u selected by `sel`, already biased to q + 128) -> fp16x2 holding
// q exactly: the byte permute builds the fp16 patterns 0x64XX = 1024 + XX.
__device__ __forceinline__ uint32_t q8_pair_to_f16x2(uint32_t u, uint32_t sel) {
    uint32_t h = __byte_perm(u, 0x64646464u, sel);
    __half2 v = *reinterpret_cast<__half2 *>(&h);
    v = __hsub2(v, __half2(__ushort_as_half(0x6480), __ushort_as_half(0x6480)));  // - 1152
    return *reinterpret_cast<uint32_t *>(&v);
}

__device__ __forceinline__ uint4 ldg_u4(const void *p) { return *reinterpret_cast<const uint4 *>(p); }

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

__device__ __forceinline__ void st_release_u32(unsigned *p, unsigned v) {
    asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// Waits (bounded) until *flag is non-zero; false if the limit ran out.
__device__ __forceinline__ bool wait_flag(const unsigned *flag, unsigned long long timeout_ns) {
    if (ld_acquire_u32(flag) != 0u) return true;
    const unsigned long long t0 = global_timer_ns();
    while (ld_acquire_u32(flag) == 0u) {
        if (global_timer_ns() - t0 > timeout_ns) return false;
        __nanosleep(64);
    }
    return true;
}

__device__ __forceinline__ void store_y(const Q8Problem &a, int row, const float (&y)[kNPad]) {
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

// Stage J is the CTA's J-th 128-k stage over all its units, in order.  Ring positions:
// shared-memory slot J % kStages, TMEM A slot and accumulator group J % kASlots, and the
// phase of each ring's barrier is (J / ring size) & 1.
template <int P, bool SK>
__global__ void __launch_bounds__(kThreads, 1) ws_q8_tc_kernel(const __grid_constant__ Q8GroupT<P> g) {
    extern __shared__ unsigned char smem_raw[];
    const uint32_t raw_addr = smem_addr(smem_raw);
    unsigned char *ring = smem_raw + ((1024u - (raw_addr & 1023u)) & 1023u);  // 1024-aligned slots
    // Barriers.  done[J % kStages] completes once per stage J when the stage's MMAs have
    // finished (one tcgen05.commit): its shared-memory slot may be refilled, its TMEM A slot
    // reused and its accumulators read.
    uint64_t *full_r = reinterpret_cast<uint64_t *>(ring + size_t(kStages) * kSlotBytes);  // TMA landed
    uint64_t *done = full_r + kStages;
    uint64_t *full_a = done + kStages;     // fp16 A tile written to TMEM (per A slot)
    uint64_t *empty_t = full_a + kASlots;  // accumulator group drained by the epilogue
    uint64_t *mma_done = empty_t + kTGroups;  // [kMmaIssuers]
    uint64_t *never = mma_done + kMmaIssuers;  // signalled by nobody: the fault-injection hook waits on it
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(never + 1);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    // TMA producer state (warp kTmaWarp, lane 0): the current piece of work (its geometry
    // computed once), stage j within it, stage J overall
    Cursor pc = cursor_begin<SK>(g);
    Unit pug;
    bool phave = cursor_next<SK>(g, pc, pug);
    int pj = 0, pJ = 0;
    bool pstop = false;
    uint64_t pol_q = 0, pol_x = 0;
    // issues the stages up to (not including) stage Jend: int8 tile + two X atoms per stage
    auto produce = [&](int Jend) {
        while (!pstop && phave && pJ < Jend) {
            if (pj >= pug.nst) {
                pj = 0;
                phave = cursor_next<SK>(g, pc, pug);
                continue;
            }
            const int st = pJ % kStages;
            // slot st was last used by stage J - kStages
            if (!mbar_wait(&done[st], static_cast<uint32_t>(((pJ / kStages) & 1) ^ 1), g.timeout_ns)) {
                atomicOr(g.status, kWsStatusTimeout);
                pstop = true;
                break;
            }
            unsigned char *slot = ring + size_t(st) * kSlotBytes;
            const int k0 = (pug.ks0 + pj) * kKS;
            mbar_arrive_expect_tx(&full_r[st], kSlotBytes);
            tma_load_3d(slot, &g.tmQ[pug.p], 0, pug.n0, k0 / 128, &full_r[st], pol_q);
            tma_load_3d(slot + kQBytes, &g.tmX[pug.p], 0, 0, k0 / 64, &full_r[st], pol_x);  // both X atoms
            ++pj;
            ++pJ;
        }
    };
    if (warp == kTmaWarp && lane == 0) {
        // The producer sets up the barriers and issues the first stages before the CTA-wide
        // set-up (TMEM allocation, the CTA barrier), so their DRAM latency overlaps it.  Two
        // only: each stage takes the producing thread ~0.2 us to issue, and a whole ring issued
        // here held the converters and MMAs back (single calls 0.6-1.7 us slower).
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&full_r[s], 1);
            mbar_init(&done[s], 1);
        }
        for (int s = 0; s < kASlots; ++s) mbar_init(&full_a[s], 4);
        for (int t = 0; t < kTGroups; ++t) mbar_init(&empty_t[t], 4);
        for (int i = 0; i < kMmaIssuers; ++i) mbar_init(&mma_done[i], 1);
        mbar_init(never, 1);
        fence_mbar_init();
        pdl_wait();  // no global-memory access before this point
        pol_q = l2_policy_evict_first();
        pol_x = l2_policy_evict_last();
        produce(kPreBarrierStages);
    }
    if (warp == kMmaWarp) tmem_alloc(tmem_slot, kTmemCols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    pdl_launch_dependents();
    pdl_wait();  // no global-memory access before this point

    if (warp == kTmaWarp) {
        // ---- TMA producer: the remaining stages ----
        if (lane == 0) {
            produce(0x7fffffff);
            // copies still in flight (possible only after a consumer gave up) land before exit
            for (int i = pJ > kStages ? pJ - kStages : 0; i < pJ; ++i)
                mbar_wait(&full_r[i % kStages], static_cast<uint32_t>((i / kStages) & 1), g.timeout_ns);
        }
    } else if (warp >= kMmaWarp) {
        // ---- MMA issuers: warp kMmaWarp + i the stages J = i mod kMmaIssuers ----
        if (lane == 0) {
            const int par = warp - kMmaWarp;
            constexpr uint32_t idesc = idesc_f16(false, kRows, kNPad);
            const uint64_t dX0 = smem_desc_sw128(smem_addr(ring + kQBytes));
            int J = 0;
            bool stop = false;
            Cursor cur = cursor_begin<SK>(g);
            Unit ug;
            while (!stop && cursor_next<SK>(g, cur, ug)) {
                const int nst = ug.nst;
                for (int j = 0; j < nst; ++j, ++J) {
                    if (J % kMmaIssuers != par) continue;
                    const int st = J % kStages, ag = J % kASlots;
                    const uint32_t ph = static_cast<uint32_t>((J / kASlots) & 1);
                    // the converters arrive on full_a only after the stage's TMA copies (X included)
                    // have landed, so this one wait orders both operands before the MMAs
                    if (!mbar_wait(&full_a[ag], ph, g.timeout_ns) || !mbar_wait(&empty_t[ag], ph ^ 1u, g.timeout_ns)) {
                        atomicOr(g.status, kWsStatusTimeout);
                        stop = true;
                        break;
                    }
                    tc_fence_after();
                    const uint64_t dB = dX0 + static_cast<uint64_t>(st * (kSlotBytes >> 4));
                    const uint32_t ta = tmem + kAColBase + static_cast<uint32_t>(ag) * kACols;
                    const uint32_t td = tmem + static_cast<uint32_t>(ag * kBlocksPerStage * kNPad);
#pragma unroll
                    for (int b = 0; b < kBlocksPerStage; ++b) {
                        // block b = k 32b .. 32b + 31: A columns 16b (+8); X atom b/2, byte offset 64 (b%2) (+32)
                        const uint64_t db = dB + static_cast<uint64_t>((b >> 1) * (kXAtomBytes >> 4) + (b & 1) * 4);
                        tc_mma_f16_ts(td + b * kNPad, ta + 16 * b, db, idesc, 0u);
                        tc_mma_f16_ts(td + b * kNPad, ta + 16 * b + 8, db + 2, idesc, 1u);
                    }
                    tc_commit(&done[st]);
                }
            }
            tc_commit(&mma_done[par]);  // arrives once every MMA this thread issued has completed
            if (!mbar_wait(&mma_done[par], 0, g.timeout_ns)) atomicOr(g.status, kWsStatusTimeout);
        }
    } else if (warp >= 4) {
        // ---- converters: one weight row's 128 int8 -> 128 fp16 in TMEM, alternate stages ----
        const int par = (warp - 4) >> 2;  // 0: even stages, 1: odd stages
        const int lg = warp & 3;          // TMEM lane quarter this warp may access
        const int r = lg * 32 + lane;     // weight row within the tile
        const uint32_t tlane = static_cast<uint32_t>(lg * 32) << 16;
        bool broken = false;
        int J = 0;
        Cursor cur = cursor_begin<SK>(g);
        Unit ug;
        while (cursor_next<SK>(g, cur, ug)) {
            const int nst = ug.nst;
            for (int j = 0; j < nst; ++j, ++J) {
                if ((J & 1) != par) continue;
                const int st = J % kStages, as = J % kASlots;
                if (!broken && !mbar_wait(&full_r[st], static_cast<uint32_t>((J / kStages) & 1), g.timeout_ns))
                    broken = true;
                if (J >= kASlots) {  // A slot J % kASlots was last read by stage J - kASlots
                    const int jp = J - kASlots;
                    if (!broken &&
                        !mbar_wait(&done[jp % kStages], static_cast<uint32_t>((jp / kStages) & 1), g.timeout_ns))
                        broken = true;
                }
                broken = __any_sync(0xffffffffu, broken);
                if (broken && lane == 0) atomicOr(g.status, kWsStatusTimeout);
                if (!broken) {
                    const unsigned char *rowp = ring + size_t(st) * kSlotBytes + r * kKS;
#pragma unroll
                    for (int h = 0; h < 2; ++h) {  // two halves of 64 k: 32 TMEM columns each
                        uint32_t v[32];
#pragma unroll
                        for (int cc = 0; cc < 4; ++cc) {
                            const int c = 4 * h + cc;  // 16-byte chunk c = k 16c .. 16c + 15, stored at c ^ (r & 7)
                            uint4 w = *reinterpret_cast<const uint4 *>(rowp + ((c ^ (r & 7)) << 4));
                            w.x ^= 0x80808080u;
                            w.y ^= 0x80808080u;
                            w.z ^= 0x80808080u;
                            w.w ^= 0x80808080u;
                            v[8 * cc + 0] = q8_pair_to_f16x2(w.x, 0x4140);
                            v[8 * cc + 1] = q8_pair_to_f16x2(w.x, 0x4342);
                            v[8 * cc + 2] = q8_pair_to_f16x2(w.y, 0x4140);
                            v[8 * cc + 3] = q8_pair_to_f16x2(w.y, 0x4342);
                            v[8 * cc + 4] = q8_pair_to_f16x2(w.z, 0x4140);
                            v[8 * cc + 5] = q8_pair_to_f16x2(w.z, 0x4342);
                            v[8 * cc + 6] = q8_pair_to_f16x2(w.w, 0x4140);
                            v[8 * cc + 7] = q8_pair_to_f16x2(w.w, 0x4342);
                        }
                        tmem_st_32(tmem + tlane + kAColBase + static_cast<uint32_t>(as) * kACols + 32u * h, v);
                    }
                    tmem_wait_st();
                    tc_fence_before();
                }
                __syncwarp();
                if (lane == 0 && !broken) mbar_arrive(&full_a[as]);
            }
        }
    } else {
        // ---- epilogue: warp w owns TMEM lanes / weight rows 32w .. 32w+31 of each unit ----
        const int lrow = warp * 32 + lane;
        if (g.stall_ns && !mbar_wait(never, 0, g.stall_ns) && threadIdx.x == 0) atomicOr(g.status, kWsStatusTimeout);
        bool ok = true;
        int J = 0;
        Cursor cur = cursor_begin<SK>(g);
        Unit ug;
        while (cursor_next<SK>(g, cur, ug)) {
            const Q8Problem &a = g.prob[ug.p];
            const int row = ug.n0 + lrow;
            const bool rowok = row < a.N;
            const uint16_t *drow = a.d + size_t(rowok ? row : 0) * (a.K / 32) + size_t(ug.sb0) * 8;
            // the row's scales, 8 per superblock, prefetched kDAhead superblocks ahead: a load
            // issued while the weight stream saturates HBM takes microseconds to return
            constexpr int kDAhead = 4;
            uint4 dq[kDAhead];
#pragma unroll
            for (int i = 0; i < kDAhead; ++i)
                dq[i] = (rowok && i < ug.nsup) ? ldg_u4(drow + size_t(i) * 8) : make_uint4(0u, 0u, 0u, 0u);
            float acc[kNPad];
#pragma unroll
            for (int m = 0; m < kNPad; ++m) acc[m] = 0.f;
            for (int s = 0; s < ug.nsup; ++s) {
                const uint32_t dw[4] = {dq[0].x, dq[0].y, dq[0].z, dq[0].w};
#pragma unroll
                for (int i = 0; i + 1 < kDAhead; ++i) dq[i] = dq[i + 1];
                dq[kDAhead - 1] = (rowok && s + kDAhead < ug.nsup) ? ldg_u4(drow + size_t(s + kDAhead) * 8)
                                                                   : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
                for (int h = 0; h < kSuper; ++h, ++J) {  // one stage = one group of 4 accumulator slots
                    const int st = J % kStages, tg = J % kTGroups;
                    if (ok) ok = mbar_wait(&done[st], static_cast<uint32_t>((J / kStages) & 1), g.timeout_ns);
                    ok = __all_sync(0xffffffffu, ok);
                    if (!ok && lane == 0) atomicOr(g.status, kWsStatusTimeout);
                    tc_fence_after();
                    const uint32_t ta = tmem + (static_cast<uint32_t>(warp * 32) << 16) +
                                        static_cast<uint32_t>(tg * kBlocksPerStage * kNPad);
                    // two blocks' sums at a time (fewer live registers); the group is handed back
                    // once all four are read
#pragma unroll
                    for (int hq = 0; hq < kBlocksPerStage; hq += 2) {
                        uint32_t v[2][16];
                        if (ok) {
                            tmem_ld_16_async(ta + hq * kNPad, v[0]);
                            tmem_ld_16_async(ta + (hq + 1) * kNPad, v[1]);
                            tmem_wait_ld();
                        } else {
#pragma unroll
                            for (int m = 0; m < kNPad; ++m) v[0][m] = v[1][m] = 0u;
                        }
                        if (hq + 2 == kBlocksPerStage) {
                            tc_fence_before();
                            __syncwarp();
                            if (lane == 0 && ok) mbar_arrive(&empty_t[tg]);
                        }
#pragma unroll
                        for (int q = 0; q < 2; ++q) {
                            const int b = h * kBlocksPerStage + hq + q;  // Q8_0 block within the superblock
                            const float dsc = __half2float(__ushort_as_half(static_cast<unsigned short>(
                                (b & 1) ? (dw[b >> 1] >> 16) : (dw[b >> 1] & 0xffffu))));
#pragma unroll
                            for (int m = 0; m < kNPad; ++m) acc[m] = fmaf(dsc, __uint_as_float(v[q][m]), acc[m]);
                        }
                    }
                }
            }
            if constexpr (SK) {
                if (ug.sb0 == 0 && ug.nsup == a.nsb) {
                    if (ok && rowok) store_y(a, row, acc);
                } else if (ug.sb0 > 0) {
                    // a later part of a row block (the first piece of this CTA's range): the
                    // partial rows go to the workspace for the CTA that holds the first part
                    float4 *pp = reinterpret_cast<float4 *>(g.partials + (size_t(blockIdx.x) * kRows + lrow) * kNPad);
#pragma unroll
                    for (int q = 0; q < kNPad / 4; ++q)
                        pp[q] = make_float4(acc[4 * q], acc[4 * q + 1], acc[4 * q + 2], acc[4 * q + 3]);
                    named_bar_sync(1, 128);  // every row of the partial written
                    if (threadIdx.x == 0 && static_cast<int>(blockIdx.x) != g.withheld_flag) {
                        __threadfence();
                        st_release_u32(g.flags + blockIdx.x, 1u);
                    }
                } else {
                    // the first part of a row block that later CTAs continue (the last piece of
                    // this CTA's range): y = p_0 + p_1 + ... in CTA order
                    const int unit_end = a.sb_base + (ug.rb + 1) * a.nsb;
                    float y[kNPad];
#pragma unroll
                    for (int m = 0; m < kNPad; ++m) y[m] = acc[m];
                    int jend = blockIdx.x + 1;
                    for (; jend < static_cast<int>(gridDim.x) && range_begin(jend, g.total_sb, gridDim.x) < unit_end;
                         ++jend) {
                        if (ok && !wait_flag(g.flags + jend, g.timeout_ns)) ok = false;
                        ok = __all_sync(0xffffffffu, ok);
                        if (!ok) {
                            if (lane == 0) atomicOr(g.status, kWsStatusTimeout);
                            continue;
                        }
                        const float4 *pp =
                            reinterpret_cast<const float4 *>(g.partials + (size_t(jend) * kRows + lrow) * kNPad);
#pragma unroll
                        for (int q = 0; q < kNPad / 4; ++q) {
                            const float4 t = pp[q];
                            y[4 * q] += t.x;
                            y[4 * q + 1] += t.y;
                            y[4 * q + 2] += t.z;
                            y[4 * q + 3] += t.w;
                        }
                    }
                    if (ok && rowok) store_y(a, row, y);
                    named_bar_sync(1, 128);  // every row has read the partials
                    if (threadIdx.x == 0 && ok)
                        for (int j = blockIdx.x + 1; j < jend; ++j) g.flags[j] = 0u;  // ready for the next launch
                }
            } else if (a.S == 1) {
                if (ok && rowok) store_y(a, row, acc);
            } else if (g.cluster) {
                // Every CTA has one unit.  First barrier: every CTA of the cluster has finished
                // its stream, so the ring of unit 0 is idle; units 1..S-1 then store this row's
                // partial into it, and after the second barrier unit 0 sums
                // y = 0 + p_0 + p_1 + ... + p_{S-1}.  Unit 0 of the row block is cluster rank
                // (c mod cluster size) - sk, the same bits whatever the cluster size.
                const int sk = ug.sk;
                const uint32_t rank0 = static_cast<uint32_t>(static_cast<int>(blockIdx.x) % g.csize - sk);
                cluster_sync_all();
                float *recv = reinterpret_cast<float *>(ring);
                if (sk != 0) {
                    const uint32_t dst = map_to_rank(smem_addr(recv + (size_t(sk - 1) * kRows + lrow) * a.mcols), rank0);
#pragma unroll
                    for (int q = 0; q < kNPad / 4; ++q)
                        if (4 * q < a.mcols)
                            st_cluster_v4(dst + 16u * q, acc[4 * q], acc[4 * q + 1], acc[4 * q + 2], acc[4 * q + 3]);
                }
                cluster_sync_all();
                if (sk == 0 && ok && rowok) {
                    float y[kNPad];
#pragma unroll
                    for (int m = 0; m < kNPad; ++m) y[m] = 0.f + acc[m];
                    for (int s2 = 1; s2 < a.S; ++s2) {
                        const float4 *src = reinterpret_cast<const float4 *>(recv + (size_t(s2 - 1) * kRows + lrow) * a.mcols);
#pragma unroll
                        for (int q = 0; q < kNPad / 4; ++q) {
                            if (4 * q < a.mcols) {
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
    }
    // cluster mode: the two barriers of the epilogue, for every other thread of the CTA
    if (!SK && g.cluster && warp >= 4 && g.prob[unit_geometry(g, blockIdx.x).p].S > 1) {
        cluster_sync_all();
        cluster_sync_all();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == kMmaWarp) tmem_dealloc(tmem, kTmemCols);
}

struct Plan {
    int nrb, nsb, S;
    bool cluster;  // one unit per CTA, the S units of a row block as one cluster
};

dspark_status configure_kernel(int dev) {
    static int configured_dev = -1;
    if (configured_dev == dev) return DSPARK_OK;
    const void *kerns[2] = {reinterpret_cast<const void *>(ws_q8_tc_kernel<1, false>),
                            reinterpret_cast<const void *>(ws_q8_tc_kernel<kMaxProblems, true>)};
    for (const void *kern : kerns) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             static_cast<int>(kSmemBytes));
        if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute(ws_matvec_q8)");
        int per_sm = 0;
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kThreads, kSmemBytes);
        if (e != cudaSuccess) return cuda_fail(e, "cudaOccupancyMaxActiveBlocksPerMultiprocessor(ws_matvec_q8)");
        if (per_sm < 1) return fail(DSPARK_ERR_CUDA, "ws_matvec_q8 kernel cannot be resident on an SM");
    }
    configured_dev = dev;
    return DSPARK_OK;
}

// How many CTAs one wave of clusters of S holds (cached per device and S).
int cluster_capacity(int S) {
    static int cache[64][kMaxSplit + 1];
    static bool init = false;
    if (!init) {
        for (auto &row : cache)
            for (int &c : row) c = -1;
        init = true;
    }
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
    if (cache[dev][S] >= 0) return cache[dev][S];
    if (configure_kernel(dev) != DSPARK_OK) return 0;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(S));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = kSmemBytes;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = static_cast<unsigned>(S);
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int c = 0;
    if (cudaOccupancyMaxActiveClusters(&c, ws_q8_tc_kernel<1, false>, &cfg) != cudaSuccess) {
        cudaGetLastError();
        c = 0;
    }
    cache[dev][S] = c * S;
    return cache[dev][S];
}

// The split of K: with at most as many row blocks as SMs, the S (1 .. kMaxSplit) that gives
// the fewest superblocks to any CTA with every unit in one wave of clusters (then the
// smaller S); each CTA takes one unit and the S units of a row block reduce in distributed
// shared memory.  More row blocks than SMs: unsplit, persistent CTAs walking the units.
Plan plan_for(int N, int K, int sms) {
    Plan p;
    p.nrb = (N + kRows - 1) / kRows;
    p.nsb = K / (kKS * kSuper);
    p.S = 1;
    p.cluster = false;
    if (p.nrb > sms) return p;
    int best = -1;
    for (int S = 1; S <= kMaxSplit && S <= p.nsb; ++S) {
        const long long units = static_cast<long long>(p.nrb) * S;
        if (units > sms) break;
        if (S > 1 && units > cluster_capacity(S)) continue;
        const int load = (p.nsb + S - 1) / S;
        if (best < 0 || load < best) {
            best = load;
            p.S = S;
        }
    }
    p.cluster = p.S > 1;
    return p;
}

__global__ void q8_0_repack_kernel(const uint8_t *__restrict__ aos, int8_t *__restrict__ q, uint16_t *__restrict__ d,
                                   long long nblocks) {
    const long long b = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (b >= nblocks) return;
    const uint8_t *src = aos + b * 34;
    d[b] = static_cast<uint16_t>(src[0] | (src[1] << 8));
    uint32_t w[8];
#pragma unroll
    for (int i = 0; i < 8; ++i)
        w[i] = src[2 + 4 * i] | (src[3 + 4 * i] << 8) | (src[4 + 4 * i] << 16) | (uint32_t(src[5 + 4 * i]) << 24);
    uint4 *dst = reinterpret_cast<uint4 *>(q + b * 32);
    dst[0] = make_uint4(w[0], w[1], w[2], w[3]);
    dst[1] = make_uint4(w[4], w[5], w[6], w[7]);
}

}  // namespace
}  // namespace dspark

extern "C" dspark_status dspark_q8_0_repack(const void *w_q8_0, int8_t *q, uint16_t *d, int N, int K,
                                            dspark_stream_t stream) {
    using namespace dspark;
    clear_error();
    if (N < 0 || K <= 0 || (K % 32) != 0) return fail(DSPARK_ERR_INVALID, "q8_0_repack: bad sizes N=%d K=%d", N, K);
    if (N == 0) return DSPARK_OK;
    if (!w_q8_0 || !q || !d) return fail(DSPARK_ERR_INVALID, "q8_0_repack: null pointer argument");
    if (!aligned(q, 16) || !aligned(d, 2)) return fail(DSPARK_ERR_INVALID, "q8_0_repack: misaligned output");
    const long long nblocks = static_cast<long long>(N) * (K / 32);
    const int threads = 256;
    const long long grid = (nblocks + threads - 1) / threads;
    q8_0_repack_kernel<<<static_cast<unsigned>(grid), threads, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
        static_cast<const uint8_t *>(w_q8_0), q, d, nblocks);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(e, "q8_0_repack launch");
    return DSPARK_OK;
}

extern "C" size_t dspark_ws_matvec_q8_workspace_bytes(int M, int N, int K) {
    // split rows reduce in distributed shared memory: the workspace holds the status word
    (void)M;
    (void)N;
    (void)K;
    return dspark::kWsHeaderBytes;
}

namespace {
using namespace dspark;

// Validation of one problem; `what` names the entry point in error texts.
dspark_status check_q8_problem(const dspark_ws_q8_problem &q, const char *what) {
    if (q.M < 0 || q.N < 0 || q.K < 0) return fail(DSPARK_ERR_INVALID, "%s: negative size", what);
    if (q.M > 16) return fail(DSPARK_ERR_UNSUPPORTED, "%s: M=%d > 16", what, q.M);
    if (q.K == 0 || (q.K % 256) != 0)
        return fail(DSPARK_ERR_UNSUPPORTED, "%s: K=%d is not a multiple of 256", what, q.K);
    if (q.M == 0 || q.N == 0) return DSPARK_OK;  // nothing to do for this problem
    if (!q.Wq || !q.Wd || !q.X || !q.Y) return fail(DSPARK_ERR_INVALID, "%s: null pointer argument", what);
    if (!aligned(q.Wq, 16) || !aligned(q.Wd, 16) || !aligned(q.X, 16))
        return fail(DSPARK_ERR_INVALID, "%s: Wq, Wd and X must be 16-byte aligned", what);
    if (!aligned(q.Y, q.y_is_fp32 ? 4 : 2)) return fail(DSPARK_ERR_INVALID, "%s: misaligned Y", what);
    return DSPARK_OK;
}

// Workspace of a grouped launch: the status header, one flag per CTA and one partial row
// block (128 rows x 16 fp32) per CTA, for at most `sms` CTAs.
size_t flags_bytes(int sms) { return (size_t(sms) * 4 + 255) / 256 * 256; }
size_t grouped_workspace_bytes(int sms) {
    return kWsHeaderBytes + flags_bytes(sms) + size_t(sms) * kRows * kNPad * sizeof(float);
}

// One launch for n problems.  A single problem keeps its own plan: one unit per CTA in
// clusters of S when it is split, else persistent CTAs walking the units.  Several problems
// run stream-K: their 128-row blocks, each over all of K, form one sequence of superblocks
// that G = min(SMs, superblocks) co-resident CTAs (a cooperative launch) take in equal
// contiguous ranges; a row block cut by a range boundary is finished by the CTA holding its
// first superblocks, which adds the partial rows of the CTAs after it in CTA order.  Every
// output is summed in one fixed order; a row block that no boundary cuts gives the same bits
// as the same problem alone without a split.  (A grid of one unit per CTA in clusters of each
// problem's split measured 41-55 us on the four Qwen3-8B projections, waves of CTAs starting
// late and tails left alone.)
dspark_status q8_enqueue_group(const dspark_ws_q8_problem *probs, int n, void *workspace, size_t workspace_bytes,
                               unsigned long long stall_ns, dspark_stream_t stream, int withheld_flag = -1,
                               unsigned long long timeout_ns = kDefaultTimeoutNs) {
    const char *what = n == 1 && probs ? "ws_matvec_q8" : "ws_matvec_q8_grouped";
    clear_error();
    if (n < 0 || n > kMaxProblems) return fail(DSPARK_ERR_UNSUPPORTED, "%s: %d problems (at most %d)", what, n, kMaxProblems);
    if (n > 0 && !probs) return fail(DSPARK_ERR_INVALID, "%s: null problem array", what);
    int live = 0;
    for (int i = 0; i < n; ++i) {
        dspark_status st = check_q8_problem(probs[i], what);
        if (st != DSPARK_OK) return st;
        if (probs[i].M != 0 && probs[i].N != 0) ++live;
    }
    if (live == 0) return DSPARK_OK;  // nothing to enqueue
    if (!workspace) return fail(DSPARK_ERR_INVALID, "%s: null workspace", what);
    if (!aligned(workspace, 256)) return fail(DSPARK_ERR_INVALID, "%s: workspace must be 256-byte aligned", what);
    if (workspace_bytes < kWsHeaderBytes)
        return fail(DSPARK_ERR_INVALID, "%s: workspace of %zu bytes < required %zu", what, workspace_bytes,
                    kWsHeaderBytes);
    int sms = 0;
    int rc = current_sm_count(&sms);
    if (rc != DSPARK_OK) return static_cast<dspark_status>(rc);
    if (live > 1 && workspace_bytes < grouped_workspace_bytes(sms))
        return fail(DSPARK_ERR_INVALID, "%s: workspace of %zu bytes < required %zu", what, workspace_bytes,
                    grouped_workspace_bytes(sms));
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    dspark_status st = configure_kernel(dev);
    if (st != DSPARK_OK) return st;

    Q8GroupT<kMaxProblems> g;
    g.nprob = 0;
    g.status = static_cast<unsigned *>(workspace);
    g.timeout_ns = timeout_ns;
    g.stall_ns = stall_ns;
    g.streamk = live > 1 ? 1 : 0;
    g.total_sb = 0;
    g.partials = nullptr;
    g.flags = nullptr;
    g.withheld_flag = withheld_flag;
    g.units = 0;
    g.csize = 1;
    g.cluster = 0;
    for (int i = 0; i < n; ++i) {
        const dspark_ws_q8_problem &q = probs[i];
        if (q.M == 0 || q.N == 0) continue;
        const int j = g.nprob++;
        st = make_tmap_kblocks_u8(&g.tmQ[j], q.Wq, static_cast<uint64_t>(q.N), static_cast<uint64_t>(q.K), kRows, 1);
        if (st != DSPARK_OK) return st;
        st = make_tmap_kblocks(&g.tmX[j], q.X, false, static_cast<uint64_t>(q.M), static_cast<uint64_t>(q.K), kNPad, 2);
        if (st != DSPARK_OK) return st;
        Q8Problem &a = g.prob[j];
        a.d = q.Wd;
        a.Y = q.Y;
        a.y_fp32 = q.y_is_fp32 ? 1 : 0;
        a.M = q.M;
        a.N = q.N;
        a.K = q.K;
        a.mcols = q.M <= 8 ? 8 : 16;
        a.unit0 = 0;
        a.sb_base = g.total_sb;
        if (g.streamk) {
            a.nrb = (q.N + kRows - 1) / kRows;
            a.nsb = q.K / (kKS * kSuper);
            a.S = 1;
            g.total_sb += a.nrb * a.nsb;
        } else {
            const Plan p = plan_for(q.N, q.K, sms);
            a.nrb = p.nrb;
            a.nsb = p.nsb;
            a.S = p.S;
            g.units = p.nrb * p.S;
            g.csize = p.cluster ? p.S : 1;
            g.cluster = p.cluster ? 1 : 0;
        }
    }
    unsigned grid;
    if (g.streamk) {
        grid = static_cast<unsigned>(g.total_sb < sms ? g.total_sb : sms);
        unsigned char *ws = static_cast<unsigned char *>(workspace);
        g.flags = reinterpret_cast<unsigned *>(ws + kWsHeaderBytes);
        g.partials = reinterpret_cast<float *>(ws + kWsHeaderBytes + flags_bytes(sms));
    } else {
        // split: one unit per CTA in clusters of S; unsplit: persistent CTAs (at most one per SM)
        grid = g.cluster ? static_cast<unsigned>(g.units)
                         : static_cast<unsigned>(g.units < sms ? g.units : sms);
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = kSmemBytes;
    cfg.stream = reinterpret_cast<cudaStream_t>(stream);
    cudaLaunchAttribute attr[2];
    cfg.attrs = attr;
    if (g.streamk) {
        // a CTA waits for the CTAs after it: all of them must be resident at once
        attr[0].id = cudaLaunchAttributeCooperative;
        attr[0].val.cooperative = 1;
        cfg.numAttrs = 1;
    } else {
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.numAttrs = 1;
        if (g.cluster) {
            attr[1].id = cudaLaunchAttributeClusterDimension;
            attr[1].val.clusterDim.x = static_cast<unsigned>(g.csize);
            attr[1].val.clusterDim.y = 1;
            attr[1].val.clusterDim.z = 1;
            cfg.numAttrs = 2;
        }
    }
    if (g.nprob == 1) {  // the small parameter block
        Q8GroupT<1> g1;
        g1.nprob = 1;
        g1.units = g.units;
        g1.cluster = g.cluster;
        g1.csize = g.csize;
        g1.streamk = g.streamk;
        g1.total_sb = g.total_sb;
        g1.partials = g.partials;
        g1.flags = g.flags;
        g1.withheld_flag = -1;
        g1.status = g.status;
        g1.timeout_ns = g.timeout_ns;
        g1.stall_ns = g.stall_ns;
        g1.prob[0] = g.prob[0];
        g1.tmQ[0] = g.tmQ[0];
        g1.tmX[0] = g.tmX[0];
        e = cudaLaunchKernelEx(&cfg, ws_q8_tc_kernel<1, false>, g1);
    } else {
        e = cudaLaunchKernelEx(&cfg, ws_q8_tc_kernel<kMaxProblems, true>, g);
    }
    if (e != cudaSuccess) return cuda_fail(e, "ws_matvec_q8 launch");
    return DSPARK_OK;
}

dspark_status q8_enqueue(const int8_t *Wq, const uint16_t *Wd, const uint16_t *X, void *Y, int y_is_fp32, int M, int N,
                         int K, void *workspace, size_t workspace_bytes, unsigned long long stall_ns,
                         dspark_stream_t stream) {
    const dspark_ws_q8_problem q = {Wq, Wd, X, Y, y_is_fp32, M, N, K};
    return q8_enqueue_group(&q, 1, workspace, workspace_bytes, stall_ns, stream);
}

}  // namespace

extern "C" dspark_status dspark_ws_matvec_q8(const int8_t *Wq, const uint16_t *Wd, const uint16_t *X, void *Y,
                                             int y_is_fp32, int M, int N, int K, void *workspace,
                                             size_t workspace_bytes, dspark_stream_t stream) {
    return q8_enqueue(Wq, Wd, X, Y, y_is_fp32, M, N, K, workspace, workspace_bytes, 0ull, stream);
}

extern "C" size_t dspark_ws_matvec_q8_grouped_workspace_bytes(const dspark_ws_q8_problem *problems, int n_problems) {
    (void)problems;
    (void)n_problems;
    int sms = 0;
    if (dspark::current_sm_count(&sms) != DSPARK_OK) return 0;
    return grouped_workspace_bytes(sms);
}

extern "C" dspark_status dspark_ws_matvec_q8_grouped(const dspark_ws_q8_problem *problems, int n_problems,
                                                     void *workspace, size_t workspace_bytes, dspark_stream_t stream) {
    return q8_enqueue_group(problems, n_problems, workspace, workspace_bytes, 0ull, stream);
}

extern "C" dspark_status dspark_ws_matvec_q8_grouped_debug(const dspark_ws_q8_problem *problems, int n_problems,
                                                           void *workspace, size_t workspace_bytes, int withheld_cta,
                                                           unsigned timeout_us, dspark_stream_t stream) {
    using namespace dspark;
    if (timeout_us == 0) return fail(DSPARK_ERR_INVALID, "ws_matvec_q8_grouped_debug: timeout_us must be > 0");
    if (withheld_cta < 0) return fail(DSPARK_ERR_INVALID, "ws_matvec_q8_grouped_debug: withheld_cta must be >= 0");
    int live = 0;
    for (int i = 0; problems && i < n_problems; ++i) live += (problems[i].M != 0 && problems[i].N != 0) ? 1 : 0;
    if (live < 2)
        return fail(DSPARK_ERR_INVALID, "ws_matvec_q8_grouped_debug: needs at least two non-empty problems");
    return q8_enqueue_group(problems, n_problems, workspace, workspace_bytes, 0ull, stream, withheld_cta,
                            1000ull * timeout_us);
}

extern "C" dspark_status dspark_ws_matvec_q8_debug(const int8_t *Wq, const uint16_t *Wd, const uint16_t *X, void *Y,
                                                   int y_is_fp32, int M, int N, int K, void *workspace,
                                                   size_t workspace_bytes, unsigned stall_us, dspark_stream_t stream) {
    if (stall_us == 0) return dspark::fail(DSPARK_ERR_INVALID, "ws_matvec_q8_debug: stall_us must be > 0");
    return q8_enqueue(Wq, Wd, X, Y, y_is_fp32, M, N, K, workspace, workspace_bytes, 1000ull * stall_us, stream);
}
