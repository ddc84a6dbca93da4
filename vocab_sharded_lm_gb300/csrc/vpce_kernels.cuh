// Kernel parameter blocks and the pipeline shape shared by the launch code
// and the kernels of the vocab-parallel cross-entropy.
#pragma once

#include "vpce_device.cuh"

namespace vpce {

// Streaming pipeline of the backward kernel: every warp owns a ring of kStages
// shared-memory slots of kChunk bytes that the bulk-copy engine fills; kWarps
// warps per block, one block per SM (persistent grid).  Measured on GB300 (s = 8192 and 32768):
// two 12 KB slots per warp beat four 6 KB ones by 6% on the backward (fewer,
// larger bulk copies for the same bytes in flight) and tie on the forward.
constexpr int kWarps = 8;
constexpr int kStages = 2;
constexpr int kChunk = 12288;
constexpr size_t kRingSmem = size_t(kWarps) * kStages * kChunk + size_t(kWarps) * kStages * sizeof(uint64_t);

// The forward statistics kernel streams into registers: kRegThreads per
// block, one warp per (shard, row) unit at a time, StatsShape<T>::kVecs
// 16-byte vectors per lane per step and kBlocksPerSm blocks per SM.
constexpr int kRegThreads = 256;
template <typename T> struct StatsShape;
template <> struct StatsShape<__nv_bfloat16> {
  static constexpr int kVecs = 16;
  static constexpr int kBlocksPerSm = 2;
};
template <> struct StatsShape<float> {
  static constexpr int kVecs = 12;
  static constexpr int kBlocksPerSm = 3;
};

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
  // The combine in the same kernel (row_cnt null: partials only).  The warp
  // that adds a row's last partial folds the row: lse[r], the row loss over
  // tgt[r], row_loss[r]; the last block to finish sums the batch.
  int* row_cnt = nullptr;   // [s] partials arrived per row, zero at launch
  int t = 0;
  long long V = 0;
  int reduction = 0;
  float* lse = nullptr;
  float* row_loss = nullptr;  // may be null
  float* loss_out = nullptr;  // may be null
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

// The units of one warp of the statistics kernel: u, u + nw, u + 2 nw,
// ... (all warps together walk the units in order, so the rows in flight at
// any time are neighbours in memory), with (shard, row) carried along.
struct WarpUnits {
  long long u, row, nw;
  int shard;
  __device__ __forceinline__ void start(long long s) {
    nw = (long long)gridDim.x * (blockDim.x >> 5);
    u = (long long)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    shard = int(u / s);
    row = u - (long long)shard * s;
  }
  __device__ __forceinline__ void next(long long s) {
    u += nw;
    row += nw;
    while (row >= s) {
      row -= s;
      ++shard;
    }
  }
};

template <typename T>
void launch_stats(const StatsParams& p, int sms, cudaStream_t st);
void launch_combine(const CombineParams& p, int blocks, cudaStream_t st);
template <typename T>
void launch_backward(const BackwardParams& p, int grid, cudaStream_t st);

}  // namespace vpce
