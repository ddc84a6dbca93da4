// Kernel parameter blocks and the pipeline shape shared by the launch code
// and the kernels of the vocab-parallel cross-entropy.
#pragma once

#include "vpce_device.cuh"

namespace vpce {

// Streaming pipeline: every warp owns a ring of kStages shared-memory slots of
// kChunk bytes that the bulk-copy engine fills; kWarps warps per block, one
// block per SM (persistent grid).  Measured on GB300 (s = 8192 and 32768):
// two 12 KB slots per warp beat four 6 KB ones by 6% on the backward (fewer,
// larger bulk copies for the same bytes in flight) and tie on the forward.
constexpr int kWarps = 8;
constexpr int kStages = 2;
constexpr int kChunk = 12288;
constexpr size_t kRingSmem = size_t(kWarps) * kStages * kChunk + size_t(kWarps) * kStages * sizeof(uint64_t);

// Forward partial statistics of every (shard, row) unit.
struct StatsParams {
  ShardSet sh;
  long long s;          // rows
  long long units;      // t * s, unit u = shard * s + row
  const long long* targets;
  long long ignore_index;
  float2* part;         // [t][s]: (local max m, sum exp(z - m))
  float* tgt;           // [s]: target logit, written by the shard that holds it
  Header* hdr;
};

// Per-row combine and the fixed-order batch reduction.
struct CombineParams {
  long long s;
  int t;
  long long V;
  const long long* targets;
  long long ignore_index;
  int reduction;
  const float2* part;
  const float* tgt;
  float* lse;
  double* bsum;
  int* bcnt;
  float* loss_out;
  float* row_loss;      // may be null
  Header* hdr;
};

// In-place backward.
struct BackwardParams {
  ShardSet sh;          // same shards, written in place
  long long s;
  long long units;
  const long long* targets;
  long long ignore_index;
  const float* lse;
  const Header* hdr;
  Header* hdr_flags;    // same header, for the timeout flag
  float grad;
  const float* grad_rows;  // [s] per-row upstream gradient, or null (use grad)
};

template <typename T>
void launch_stats(const StatsParams& p, int grid, cudaStream_t st);
void launch_combine(const CombineParams& p, int blocks, cudaStream_t st);
template <typename T>
void launch_backward(const BackwardParams& p, int grid, cudaStream_t st);

}  // namespace vpce
