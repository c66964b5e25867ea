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
// Grid of the Markov kernel for a vocabulary of V rows on `sms` SMs: the fewest CTAs whose
// largest share of 128-row tiles equals that of an even split over all SMs.
int markov_grid(int V, int sms);

// Workspace bytes for k positions, and the checked enqueue behind every Markov entry point
// (markov.cu): memset of the workspace header + the cooperative kernel, on `stream`; with
// clear_out_ids, out_ids is first set to -1.
size_t workspace_bytes(int k);
dspark_status markov_enqueue(const float *base, const uint16_t *w1, const uint16_t *w2, const int32_t *d2t,
                             int64_t *prev, int B, int k, int V, int R, int64_t *out_ids, float *dbg_logits,
                             float *dbg_bias, void *workspace, size_t ws_bytes, unsigned bar_extra,
                             unsigned long long timeout_ns, cudaStream_t stream, bool clear_out_ids = false);

}  // namespace dspark
