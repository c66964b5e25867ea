// Shared definitions of the Markov block-draft kernels (CUDA-core and tcgen05 forms).
#pragma once

#include "common.cuh"

namespace dspark {

constexpr int kMaxReqs = 8;
constexpr size_t kHeaderBytes = 256;  // workspace header: [0] barrier arrivals, [1] status bits

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

// tcgen05 form (markov_tc.cu): at most one CTA per SM, cooperative launch.
dspark_status launch_markov_tc(const MarkovArgs &args, int R, int nctas, cudaStream_t stream);
// Single-cluster form (markov_cluster.cu): the cluster size C for B requests over a
// vocabulary of V rows of rank R and k positions on the current device, or 0 when its
// shared memory (markov_w1 and markov_w2 tiles, base rows, the exchange buffers) does not
// fit in one cluster (or V is not a multiple of 4).  Its ids and logits are bit-identical
// to the grid form's.  The launch needs a 16-byte aligned base and resets the status word
// itself (no workspace memset).
int markov_cluster_size(int B, int V, int R, int k);
dspark_status launch_markov_cluster(const MarkovArgs &args, int R, int C, cudaStream_t stream);

// Kernel choice of markov_enqueue (values of DSPARK_MARKOV_KERNEL_* in dspark.h).
constexpr int kMarkovAuto = 0;
constexpr int kMarkovGrid = 1;
constexpr int kMarkovCluster = 2;
// The kernel kMarkovAuto picks: the single-cluster form where it applies and num_reqs is at
// most kMarkovClusterAutoMaxReqs, else the grid.
constexpr int kMarkovClusterAutoMaxReqs = 2;
int markov_auto_kernel(const float *base, int B, int V, int R, int k);
// Grid of the Markov kernel for a vocabulary of V rows on `sms` SMs: the fewest CTAs whose
// largest share of 128-row tiles equals that of an even split over all SMs.
int markov_grid(int V, int sms);

// Workspace bytes for k positions, and the checked enqueue behind every Markov entry point
// (markov.cu), on `stream`: the grid form is a memset of the workspace header + the
// cooperative kernel, the cluster form its kernel alone; with clear_out_ids, out_ids is first
// set to -1.  `kernel` is kMarkovAuto, kMarkovGrid or kMarkovCluster (DSPARK_ERR_UNSUPPORTED
// when the cluster form does not apply).
size_t workspace_bytes(int k);
dspark_status markov_enqueue(const float *base, const uint16_t *w1, const uint16_t *w2, const int32_t *d2t,
                             int64_t *prev, int B, int k, int V, int R, int64_t *out_ids, float *dbg_logits,
                             float *dbg_bias, void *workspace, size_t ws_bytes, unsigned bar_extra,
                             unsigned long long timeout_ns, cudaStream_t stream, bool clear_out_ids = false,
                             int kernel = kMarkovAuto);

}  // namespace dspark
