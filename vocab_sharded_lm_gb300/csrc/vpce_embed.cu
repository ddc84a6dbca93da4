// Vocabulary-parallel input embedding, forward and backward.
//
// "Distributed Training III: Model Parallelism" (CMU 11-868 Lecture 16 notes),
// §5.5, and "LLM Internals" §7.3.4: the table [V, h] is split by vocabulary
// into t shards; card i looks up only the ids in its range, writes zeros
// elsewhere, and an all-reduce sums the cards.  With every shard on one GPU
// the sum has exactly one non-zero term per row, so the forward is a gather
// of that term: each warp finds the shard that holds its row's id and copies
// the row (16-byte vectors, streaming loads); an id in no shard's range
// gives a zero row and raises a flag bit.
//
// The backward (not on the pages; the adjoint of the lookup) adds each
// output-gradient row into the table row of its id.  It is deterministic and
// takes two launches per chunk of up to kEmbChunk rows: a cluster of eight
// CTAs sorts the chunk's (id, row) pairs (bitonic within each CTA, then
// merge-path rounds through distributed shared memory) and marks where each
// id's run starts, listing the long runs and grouping the short ones; one
// persistent kernel then sums every run in a fixed order and adds the sum
// into the fp32 gradient table, streaming the rows through shared memory with
// cp.async.  Longer batches run chunk after chunk on the stream, so the
// accumulation order is fixed.
#include <cooperative_groups.h>

#include "vpce_kernels.cuh"

namespace vpce {

namespace {

constexpr int kEmbThreads = 256;
constexpr int kSortThreads = 1024;
constexpr int kEmbChunk = 16384;  // rows sorted per backward chunk (128 KB of keys)
constexpr int kHeavyRows = 64;  // ids with more rows are summed by a whole CTA
constexpr int kGroupRows = 16;  // short-run tasks: runs starting in this many consecutive sorted rows

struct EmbedFwdParams {
  ShardSet sh;        // table shards [w_i, h] (ld_bytes = row stride)
  int t;
  long long V;
  long long h;        // columns
  int eb;             // element bytes (2 or 4)
  const long long* ids;
  long long s;
  unsigned char* out;
  long long ld_out_bytes;
  int* flag;          // may be null
};

// shard that holds id (-1: none)
__device__ __forceinline__ int shard_of(const long long* start, int t, long long id) {
  if (id < start[0] || id >= start[t]) return -1;
  int lo = 0, hi = t;  // start[lo] <= id < start[hi]
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (start[mid] <= id) lo = mid;
    else hi = mid;
  }
  return lo;
}

__global__ void __launch_bounds__(kEmbThreads) embed_forward_kernel(const __grid_constant__ EmbedFwdParams p) {
  __shared__ long long start[VPCE_MAX_SHARDS + 1];
  __shared__ const unsigned char* base[VPCE_MAX_SHARDS];
  __shared__ long long ldb[VPCE_MAX_SHARDS];
  for (int i = threadIdx.x; i <= p.t; i += kEmbThreads) {
    start[i] = p.sh.start[i];
    if (i < p.t) {
      base[i] = p.sh.ptr[i];
      ldb[i] = p.sh.ld_bytes[i];
    }
  }
  __syncthreads();
  const int lane = threadIdx.x & 31;
  const long long row_bytes = p.h * p.eb;
  const long long nwarps = (long long)gridDim.x * (kEmbThreads / 32);
  for (long long r = (long long)blockIdx.x * (kEmbThreads / 32) + (threadIdx.x >> 5); r < p.s; r += nwarps) {
    const long long id = p.ids[r];
    const int i = shard_of(start, p.t, id);
    unsigned char* dst = p.out + r * p.ld_out_bytes;
    const unsigned char* src = i >= 0 ? base[i] + (id - start[i]) * ldb[i] : nullptr;
    const bool vec = ((reinterpret_cast<uintptr_t>(dst) | reinterpret_cast<uintptr_t>(src) | row_bytes) & 15) == 0;
    if (i < 0 && lane == 0 && p.flag != nullptr) atomicOr(p.flag, VPCE_FLAG_BAD_TARGET);
    if (vec) {
      const long long nv = row_bytes >> 4;
      uint4* d = reinterpret_cast<uint4*>(dst);
      const uint4* sp = reinterpret_cast<const uint4*>(src);
      long long v = lane;
      // eight independent 16-byte streaming loads in flight per lane (plain
      // intrinsics, so the compiler may also start the next eight early)
      for (; v + 224 < nv; v += 256) {
        uint4 q[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) q[u] = i >= 0 ? __ldcs(sp + v + 32 * u) : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
        for (int u = 0; u < 8; ++u) d[v + 32 * u] = q[u];
      }
      for (; v < nv; v += 32) d[v] = i >= 0 ? __ldcs(sp + v) : make_uint4(0u, 0u, 0u, 0u);
    } else if (p.eb == 2) {
      unsigned short* d = reinterpret_cast<unsigned short*>(dst);
      const unsigned short* sp = reinterpret_cast<const unsigned short*>(src);
      for (long long c = lane; c < p.h; c += 32) d[c] = i >= 0 ? sp[c] : (unsigned short)0;
    } else {
      unsigned* d = reinterpret_cast<unsigned*>(dst);
      const unsigned* sp = reinterpret_cast<const unsigned*>(src);
      for (long long c = lane; c < p.h; c += 32) d[c] = i >= 0 ? sp[c] : 0u;
    }
  }
}

// ---------------------------------------------------------------------------
// backward
// ---------------------------------------------------------------------------
constexpr int kSortCtas = 8;                        // one thread-block cluster per chunk
constexpr int kSortKeys = kEmbChunk / kSortCtas;    // keys per CTA, at most
constexpr int kMaxHeavyPerCta = kSortKeys / (kHeavyRows + 1) + 1;

// Sort keys (id << kShift | row): 32 bits when the ids and a chunk's rows fit
// (ids below 2^18 - 2, rows below 2^14), 64 otherwise; kNone (padding and
// ids outside [0, V)) sorts after every valid key.
template <typename K>
struct SortKey;
template <>
struct SortKey<unsigned> {
  static constexpr int kShift = 14;
  static constexpr unsigned kNone = 0xffffffffu;
};
template <>
struct SortKey<unsigned long long> {
  static constexpr int kShift = 32;
  static constexpr unsigned long long kNone = ~0ull;
};
static_assert(kEmbChunk <= (1 << 14), "rows of a chunk fit the 32-bit key");
constexpr long long kMaxV32 = (1LL << 18) - 2;  // vocabularies up to this size use 32-bit keys

struct EmbedSortParams {
  const long long* ids;            // this chunk's ids
  int n;                           // ids in the chunk
  int n_pow2;                      // a power of two >= n and >= kSortCtas
  long long V;
  int* rows;                       // [n_pow2] out: the rows in (id, row) order, -1 for the padding last
  int* seg;                        // [kEmbChunk + 1] start of each distinct id's run; seg[n_seg] = valid keys
  int* heavy;                      // runs longer than kHeavyRows (any order)
  int* gstart;                     // [kEmbChunk / kGroupRows + 1] first run of each group of kGroupRows rows
  unsigned long long* rtab;        // [kEmbChunk] each run's gradient-table row (address)
  int* counts;                     // n_seg, n_heavy, n_grp, work[2] (the accumulation's counters, cleared)
  Header* hdr;                     // error flag (cleared when `first`)
  int first;                       // first chunk of the call
  ShardSet gsh;                    // fp32 gradient table shards
  int t;
};

// Exclusive scan of one int per thread in thread order; *total gets the sum.
__device__ __forceinline__ int block_scan(int v, int* warp_tmp, int* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int x = __shfl_up_sync(kFull, incl, o);
    if (lane >= o) incl += x;
  }
  if (lane == 31) warp_tmp[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    int w = lane < int(blockDim.x >> 5) ? warp_tmp[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int x = __shfl_up_sync(kFull, w, o);
      if (lane >= o) w += x;
    }
    warp_tmp[lane] = w;  // inclusive over warps
  }
  __syncthreads();
  const int ex = incl - v + (warp > 0 ? warp_tmp[warp - 1] : 0);
  *total = warp_tmp[(blockDim.x >> 5) - 1];
  __syncthreads();
  return ex;
}

// One chunk's sort and run scan in one launch: a cluster of kSortCtas CTAs,
// each holding B = n_pow2 / kSortCtas keys.
//  1. CTA c builds the (id, row) keys of rows [c B, (c + 1) B) (kNone for
//     padding and for ids outside [0, V)) and bitonic-sorts them in shared
//     memory.
//  2. One multiway merge: every CTA copies the other blocks from distributed
//     shared memory, and a key's place is its index in its block plus its
//     rank in each other block (blocks before c count keys <= it, blocks
//     after count keys < it, so equal padding keys keep block order); the key
//     is stored straight into the shared memory of the CTA that owns that
//     place.
//  3. The run heads (a valid key whose id differs from its predecessor's),
//     numbered by a scan over the cluster, give the run starts; then each run's
//     table row, the groups' first runs and the list of long runs.
template <typename K>
__global__ void __cluster_dims__(kSortCtas, 1, 1) __launch_bounds__(kSortThreads, 1)
    embed_sort_runs_kernel(const __grid_constant__ EmbedSortParams p) {
  namespace cg = cooperative_groups;
  using KT = SortKey<K>;
  cg::cluster_group cluster = cg::this_cluster();
  extern __shared__ __align__(16) unsigned char sort_raw[];  // [kSortCtas * B] blocks, then [B] sorted
  __shared__ int warp_tmp[32];
  __shared__ int tot[3];  // this CTA's valid keys, run heads, long runs
  __shared__ int sh[4];   // head offset, total heads, valid keys, long-run offset
  __shared__ int hcount;
  __shared__ int hl[kMaxHeavyPerCta];
  __shared__ long long start[VPCE_MAX_SHARDS + 1];
  const int c = int(cluster.block_rank());
  const int tid = threadIdx.x;
  const int B = p.n_pow2 / kSortCtas;
  K* blocks = reinterpret_cast<K*>(sort_raw);
  K* mine = blocks + c * B;
  K* sorted = blocks + kSortCtas * B;
  for (int i = tid; i <= p.t; i += kSortThreads) start[i] = p.gsh.start[i];
  for (int k = tid; k < B; k += kSortThreads) {
    const int g = c * B + k;
    K v = KT::kNone;
    if (g < p.n) {
      const long long id = p.ids[g];
      if (id >= 0 && id < p.V) v = (static_cast<K>(id) << KT::kShift) | K(g);
    }
    mine[k] = v;
  }
  if (tid == 0) hcount = 0;
  __syncthreads();
  if (B <= kSortThreads) {
    // one key per thread: strides below 32 exchange by shuffle, larger ones
    // through shared memory (thread t >= B holds padding nobody reads)
    K x = tid < B ? mine[tid] : KT::kNone;
    for (int size = 2; size <= B; size <<= 1) {
      for (int stride = size >> 1; stride > 0; stride >>= 1) {
        K y;
        if (stride >= 32) {
          __syncthreads();  // the previous exchange's reads are done
          if (tid < B) mine[tid] = x;
          __syncthreads();
          y = tid < B ? mine[tid ^ stride] : KT::kNone;
        } else {
          y = __shfl_xor_sync(kFull, x, stride);
        }
        const bool up = (tid & size) == 0, low = (tid & stride) == 0;
        x = low == up ? (x < y ? x : y) : (x < y ? y : x);
      }
    }
    __syncthreads();
    if (tid < B) mine[tid] = x;
  } else {
    for (int size = 2; size <= B; size <<= 1) {
      for (int stride = size >> 1; stride > 0; stride >>= 1) {
        for (int k = tid; k < B / 2; k += kSortThreads) {
          const int lo = 2 * k - (k & (stride - 1));  // first element of this compare pair
          const int hi = lo + stride;
          const bool up = (lo & size) == 0;
          const K x = mine[lo], y = mine[hi];
          if ((x > y) == up) {
            mine[lo] = y;
            mine[hi] = x;
          }
        }
        __syncthreads();
      }
    }
  }
  cluster.sync();  // every block is sorted
  for (int i = tid; i < kSortCtas * B; i += kSortThreads) {
    const int r = i / B;
    if (r != c) blocks[i] = *cluster.map_shared_rank(&blocks[i], r);
  }
  __syncthreads();
  // rank of key v in block r: the keys of block r before v in the merged
  // order (blocks before c: keys <= v; after c: keys < v), searched in
  // [lo, hi] (the rank is known to lie there) in lockstep steps of p, p/2, .., 1
  auto before = [&](int r, K x, K v) { return r < c ? (x <= v) : (x < v); };
  const int lane = tid & 31;
  for (int k = tid; k < B; k += kSortThreads) {
    const K v = mine[k];
    int lo[kSortCtas], hi[kSortCtas];
#pragma unroll
    for (int r = 0; r < kSortCtas; ++r) {
      lo[r] = 0;
      hi[r] = B;
    }
    if (B >= 32) {
      // the warp's 32 keys are consecutive: lanes 0..13 find the ranks of the
      // first and the last of them in the 7 other blocks, which bound every
      // lane's rank
      const int k0 = k - lane;
      const int which = lane & 1, oth = lane >> 1;  // other block number oth (skipping c)
      const int rb = oth < c ? oth : oth + 1;
      int pos = 0;
      if (lane < 2 * (kSortCtas - 1)) {
        const K ve = mine[k0 + (which ? 31 : 0)];
        for (int step = B; step >= 1; step >>= 1)
          if (pos + step <= B && before(rb, blocks[rb * B + pos + step - 1], ve)) pos += step;
      }
#pragma unroll
      for (int j = 0; j < kSortCtas - 1; ++j) {
        const int r = j < c ? j : j + 1;  // warp-uniform
        const int l = __shfl_sync(kFull, pos, 2 * j), h = __shfl_sync(kFull, pos, 2 * j + 1);
#pragma unroll
        for (int rr = 0; rr < kSortCtas; ++rr)
          if (rr == r) {
            lo[rr] = l;
            hi[rr] = h;
          }
      }
    }
    int span = 0;
#pragma unroll
    for (int r = 0; r < kSortCtas; ++r) span = r == c ? span : max(span, hi[r] - lo[r]);
    int p2 = 1;
    while (p2 < span) p2 <<= 1;
    int o = k;
#pragma unroll
    for (int r = 0; r < kSortCtas; ++r) {
      if (r == c) continue;
      int pos = lo[r];
      for (int step = p2; step >= 1; step >>= 1)
        if (pos + step <= hi[r] && before(r, blocks[r * B + pos + step - 1], v)) pos += step;
      o += pos;
    }
    *cluster.map_shared_rank(&sorted[o % B], o / B) = v;
  }
  cluster.sync();  // the sorted keys: rows [c B, (c + 1) B) in CTA c's `sorted`
  const K* key = sorted;
  for (int k = tid; k < B; k += kSortThreads)
    p.rows[c * B + k] = key[k] == KT::kNone ? -1 : int(key[k] & ((K(1) << KT::kShift) - 1));
  const K prev_last = c > 0 ? *cluster.map_shared_rank(&sorted[B - 1], c - 1) : KT::kNone;
  const int per = (B + kSortThreads - 1) / kSortThreads;  // this thread's keys: [k0, k0 + per)
  const int k0 = tid * per;
  auto is_head = [&](int k) {
    const K v = key[k];
    if (v == KT::kNone) return false;
    if (c == 0 && k == 0) return true;
    const K pv = k > 0 ? key[k - 1] : prev_last;  // valid: valid keys come first
    return (pv >> KT::kShift) != (v >> KT::kShift);
  };
  int nv = 0, nh = 0;
  for (int k = k0; k < k0 + per && k < B; ++k) {
    nv += key[k] != KT::kNone;
    nh += is_head(k);
  }
  int vtot, htot;
  block_scan(nv, warp_tmp, &vtot);
  const int hex = block_scan(nh, warp_tmp, &htot);
  if (tid == 0) {
    tot[0] = vtot;
    tot[1] = htot;
  }
  cluster.sync();
  if (tid == 0) {
    int hoff = 0, total = 0, nvalid = 0;
    for (int r = 0; r < kSortCtas; ++r) {
      const int* rt = cluster.map_shared_rank(tot, r);
      const int hr = rt[1];
      if (r < c) hoff += hr;
      total += hr;
      nvalid += rt[0];
    }
    sh[0] = hoff;
    sh[1] = total;
    sh[2] = nvalid;
  }
  __syncthreads();
  const int total = sh[1], nvalid = sh[2];
  int j = sh[0] + hex;
  for (int k = k0; k < k0 + per && k < B; ++k)
    if (is_head(k)) p.seg[j++] = c * B + k;
  if (c == 0 && tid == 0) p.seg[total] = nvalid;
  cluster.sync();  // every run start is in global memory
  const int ngrp = (nvalid + kGroupRows - 1) / kGroupRows;
  j = sh[0] + hex;
  for (int k = k0; k < k0 + per && k < B; ++k) {
    if (!is_head(k)) continue;
    const int a = c * B + k, b = p.seg[j + 1];
    if (b - a > kHeavyRows) hl[atomicAdd(&hcount, 1)] = j;
    const long long id = static_cast<long long>(key[k] >> KT::kShift);
    const int i = shard_of(start, p.t, id);
    p.rtab[j] = reinterpret_cast<unsigned long long>(p.gsh.ptr[i] + (id - start[i]) * p.gsh.ld_bytes[i]);
    // groups g with g kGroupRows in (previous run start, a] begin with run j
    const int g_lo = j == 0 ? 0 : p.seg[j - 1] / kGroupRows + 1;
    for (int g = g_lo; g <= a / kGroupRows; ++g) p.gstart[g] = j;
    if (j == total - 1)  // groups after the last run start are empty
      for (int g = a / kGroupRows + 1; g <= ngrp; ++g) p.gstart[g] = total;
    ++j;
  }
  if (total == 0 && c == 0 && tid == 0) p.gstart[0] = 0;
  __syncthreads();
  if (tid == 0) tot[2] = hcount;
  cluster.sync();
  if (tid == 0) {
    int off = 0, nheavy = 0;
    for (int r = 0; r < kSortCtas; ++r) {
      const int hr = cluster.map_shared_rank(tot, r)[2];
      if (r < c) off += hr;
      nheavy += hr;
    }
    sh[3] = off;
    if (c == 0) {
      p.counts[0] = total;
      p.counts[1] = nheavy;
      p.counts[2] = ngrp;
      p.counts[3] = 0;  // the accumulation's task counters
      p.counts[4] = 0;
      if (p.first) p.hdr->error_flag = 0;
    }
  }
  __syncthreads();
  for (int i = tid; i < hcount; i += kSortThreads) p.heavy[sh[3] + i] = hl[i];
  cluster.sync();  // no CTA leaves while another may still read its shared memory
}

struct EmbedAccParams {
  const int* rows;  // the chunk's rows in (id, row) order
  const int* seg;
  const int* n_seg;
  const int* heavy;
  const int* n_heavy;
  const unsigned char* grad;  // this chunk's output-gradient rows
  long long ld_grad_bytes;
  int grad_bf16;
  long long h;
  ShardSet gsh;  // fp32 gradient table shards (ld_bytes = row stride)
  int t;
  const int* gstart;
  const int* n_grp;
  const unsigned long long* rtab;  // each run's gradient-table row
  unsigned* work;                  // [2] task counters (zero at launch)
  Header* hdr;
};

__device__ __forceinline__ void cp_async16(void* smem, const void* gmem, unsigned src_bytes) {
  // src_bytes < 16 zero-fills the rest of the 16 bytes
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(smem_addr(smem)), "l"(gmem), "r"(src_bytes)
               : "memory");
}
// the mbarrier receives this thread's arrival once all its earlier cp.async
// copies have landed
__device__ __forceinline__ void cp_async_arrive(uint64_t* bar) {
  asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(smem_addr(bar)) : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

constexpr int kAWarps = 8;
constexpr int kAThreads = kAWarps * 32;
constexpr int kShortCols = 256;  // columns per short-run task (8 per lane)
constexpr int kHeavyCols = 256;  // columns per long-run CTA task (8 per lane)
constexpr int kTRing = 8;        // runs (table slices) in flight per warp, at most 32

// A lane's share of a row slice of COLS columns, staged as 16-byte pieces:
// piece pc of lane l starts at column c0 + (32 pc + l) 16 / EB, so that a
// warp's piece pc is one contiguous span.  The lane's columns form COLS / 128
// quads of four (the fp32 table side): a bf16 piece holds quads 2 pc and
// 2 pc + 1, an fp32 piece is one quad.  Accumulator acc[4 q + e] is column e
// of quad q.
template <int EB, int COLS>
struct Slice {
  static constexpr int kPieces = COLS * EB / 512;
  static constexpr int kQuads = COLS / 128;
  static __device__ __forceinline__ long long piece_col(long long c0, int lane, int pc) {
    return c0 + (32LL * pc + lane) * (16 / EB);
  }
  static __device__ __forceinline__ long long quad_col(long long c0, int lane, int qd) {
    return EB == 2 ? c0 + 8 * lane + 4 * (qd & 1) + 256 * (qd >> 1) : c0 + 4 * lane + 128 * qd;
  }
};

template <int EB>
struct AccCfg {
  static constexpr int kRingBytes = EB == 2 ? 4096 : 8192;  // per warp, shared by both phases
  static constexpr int kRS = kRingBytes / (kShortCols * EB);  // short-run row slices in flight
  static constexpr int kRH = kRingBytes / (kHeavyCols * EB);  // long-run row slices in flight
};

template <int EB>
struct AccSmem {
  uint4 ring[kAWarps][AccCfg<EB>::kRingBytes / 16];  // slot-major: [slot][piece][lane]
  float4 table[kAWarps][kTRing][kShortCols / 128][32];
  float4 part[kAWarps][kHeavyCols / 128][32];
  uint64_t bar_s[kAWarps][AccCfg<EB>::kRS];
  uint64_t bar_h[kAWarps][AccCfg<EB>::kRH];
  unsigned task;
};

// A lane's view of 64 consecutive entries of an array, starting at a
// warp-uniform index that only moves forward: entries base + lane and
// base + 32 + lane, so that the next 32 are already on their way.
template <typename T>
struct Window {
  const T* a;
  long long n;  // entries [0, n) exist
  long long base;
  T cur, nxt;
  __device__ __forceinline__ T ld(long long i) const { return i < n ? a[i] : T(0); }
  __device__ __forceinline__ void init(const T* arr, long long len, long long k, int lane) {
    a = arr;
    n = len;
    base = k;
    cur = ld(k + lane);
    nxt = ld(k + 32 + lane);
  }
  __device__ __forceinline__ T at(long long k, int lane) {  // k >= base, warp-uniform
    if (k - base >= 64) {
      base = k;
      cur = ld(k + lane);
      nxt = ld(k + 32 + lane);
    } else if (k - base >= 32) {
      base += 32;
      cur = nxt;
      nxt = ld(base + 32 + lane);
    }
    return __shfl_sync(kFull, cur, int(k - base));
  }
  // entries k and k + 1, leaving the window at or before k
  __device__ __forceinline__ void pair(long long k, int lane, T& v0, T& v1) {
    const T a0 = at(k, lane);
    const int d = int(k - base);
    const T c1 = __shfl_sync(kFull, cur, (d + 1) & 31);
    const T n0 = __shfl_sync(kFull, nxt, 0);
    v0 = a0;
    v1 = d < 31 ? c1 : n0;
  }
};

// One lane's cp.async copies of one row slice into ring slot `slot`, and its
// arrival on the slot's mbarrier once they land.  Columns at or past h are
// zero-filled, nothing is read there.
template <int EB, int COLS>
__device__ __forceinline__ void stage_row(uint4* ring, int slot, int lane, const unsigned char* grow, long long c0,
                                          long long h, uint64_t* bar) {
  using S = Slice<EB, COLS>;
#pragma unroll
  for (int pc = 0; pc < S::kPieces; ++pc) {
    const long long col = S::piece_col(c0, lane, pc);
    const long long left = (h - col) * EB;
    const unsigned bytes = left >= 16 ? 16u : (left > 0 ? unsigned(left) : 0u);
    cp_async16(&ring[(slot * S::kPieces + pc) * 32 + lane], bytes ? grow + col * EB : grow, bytes);
  }
  cp_async_arrive(bar);
}

// acc += the lane's share of the row slice in ring slot `slot`
template <int EB, int COLS>
__device__ __forceinline__ void add_row(const uint4* ring, int slot, int lane, float* acc) {
  using S = Slice<EB, COLS>;
#pragma unroll
  for (int pc = 0; pc < S::kPieces; ++pc) {
    const uint4 v = ring[(slot * S::kPieces + pc) * 32 + lane];
    if (EB == 2) {
      float* a = acc + 8 * pc;
      a[0] += bf16_lo(v.x);
      a[1] += bf16_hi(v.x);
      a[2] += bf16_lo(v.y);
      a[3] += bf16_hi(v.y);
      a[4] += bf16_lo(v.z);
      a[5] += bf16_hi(v.z);
      a[6] += bf16_lo(v.w);
      a[7] += bf16_hi(v.w);
    } else {
      float* a = acc + 4 * pc;
      a[0] += __uint_as_float(v.x);
      a[1] += __uint_as_float(v.y);
      a[2] += __uint_as_float(v.z);
      a[3] += __uint_as_float(v.w);
    }
  }
}

// Every run's sum, added into its id's row of the fp32 gradient table, in
// one persistent launch.  Work is handed out through two counters.  First
// the long runs (more than kHeavyRows rows): one CTA per (run, kHeavyCols
// columns), each warp summing a contiguous eighth of the run and warp 0
// adding the eight partials in warp order.  Then the short runs: one warp
// per (group of the runs that start in kGroupRows consecutive sorted rows,
// kShortCols columns).  A warp streams its rows through a shared-memory
// ring: each lane copies its own 16-byte pieces with cp.async and the copy
// of the next row is issued as soon as a slot frees, across run boundaries;
// a run's table slice comes in with its first row, and the sum of the run's
// rows, in ascending order, is added to it after the run's last row.  Each
// element's sum has a fixed order whichever CTA or warp does the task.
template <int EB>
__global__ void __launch_bounds__(kAThreads) embed_accum_kernel(const __grid_constant__ EmbedAccParams p) {
  using C = AccCfg<EB>;
  using SS = Slice<EB, kShortCols>;
  using SH = Slice<EB, kHeavyCols>;
  extern __shared__ __align__(16) unsigned char smem_raw[];
  AccSmem<EB>& sm = *reinterpret_cast<AccSmem<EB>*>(smem_raw);
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  uint4* ring = sm.ring[w];
  if (lane == 0) {
    for (int k = 0; k < C::kRS; ++k) mbar_init(&sm.bar_s[w][k], 32);
    for (int k = 0; k < C::kRH; ++k) mbar_init(&sm.bar_h[w][k], 32);
    fence_mbar_init();
  }
  __syncthreads();
  const long long h = p.h;
  const int total = *p.n_seg;
  const long long nkeys = p.seg[total];  // valid keys
  bool ok = true;

  // ---- long runs: CTA tasks
  {
    const long long ncb = (h + kHeavyCols - 1) / kHeavyCols;
    const long long n_ht = (long long)(*p.n_heavy) * ncb;
    unsigned issued = 0, consumed = 0;
    for (;;) {
      if (threadIdx.x == 0) sm.task = atomicAdd(&p.work[0], 1u);
      __syncthreads();
      const long long q = sm.task;
      __syncthreads();
      if (q >= n_ht) break;
      const long long hj = q / ncb;
      const long long c0 = (q - hj * ncb) * kHeavyCols;
      const int sgi = p.heavy[hj];
      const int ra = p.seg[sgi], n = p.seg[sgi + 1] - ra;
      const int lo = ra + int((long long)n * w / kAWarps), hi = ra + int((long long)n * (w + 1) / kAWarps);
      float* trow = nullptr;
      float4 tq[SH::kQuads];
#pragma unroll
      for (int qd = 0; qd < SH::kQuads; ++qd) tq[qd] = make_float4(0.f, 0.f, 0.f, 0.f);
      if (w == 0) {
        trow = reinterpret_cast<float*>(p.rtab[sgi]);
#pragma unroll
        for (int qd = 0; qd < SH::kQuads; ++qd) {
          const long long col = SH::quad_col(c0, lane, qd);
          if (col < h) tq[qd] = *reinterpret_cast<const float4*>(trow + col);
        }
      }
      float acc[4 * SH::kQuads];
#pragma unroll
      for (int e = 0; e < 4 * SH::kQuads; ++e) acc[e] = 0.f;
      Window<int> kw;
      kw.init(p.rows, nkeys, lo, lane);
      long long pk = lo;
      for (int k = lo; k < hi && ok; ++k) {
        while (pk < hi && issued - consumed < unsigned(C::kRH)) {
          const int row = kw.at(pk++, lane);
          const int slot = int(issued % C::kRH);
          stage_row<EB, kHeavyCols>(ring, slot, lane, p.grad + (long long)row * p.ld_grad_bytes, c0, h,
                                    &sm.bar_h[w][slot]);
          ++issued;
        }
        const int slot = int(consumed % C::kRH);
        ok = mbar_wait_warp(&sm.bar_h[w][slot], (consumed / C::kRH) & 1u);
        if (ok) add_row<EB, kHeavyCols>(ring, slot, lane, acc);
        ++consumed;
      }
#pragma unroll
      for (int qd = 0; qd < SH::kQuads; ++qd)
        sm.part[w][qd][lane] = make_float4(acc[4 * qd], acc[4 * qd + 1], acc[4 * qd + 2], acc[4 * qd + 3]);
      __syncthreads();
      if (w == 0) {
#pragma unroll
        for (int qd = 0; qd < SH::kQuads; ++qd) {
          const long long col = SH::quad_col(c0, lane, qd);
          if (col >= h) continue;
          float4 tot = sm.part[0][qd][lane];
#pragma unroll
          for (int ww = 1; ww < kAWarps; ++ww) {
            const float4 v = sm.part[ww][qd][lane];
            tot.x += v.x;
            tot.y += v.y;
            tot.z += v.z;
            tot.w += v.w;
          }
          tq[qd].x += tot.x;
          tq[qd].y += tot.y;
          tq[qd].z += tot.z;
          tq[qd].w += tot.w;
          *reinterpret_cast<float4*>(trow + col) = tq[qd];
        }
      }
      __syncthreads();
    }
  }

  // ---- short runs: warp tasks
  const long long ncb = (h + kShortCols - 1) / kShortCols;
  const long long n_st = (long long)(*p.n_grp) * ncb;
  unsigned issued = 0, consumed = 0, run_ord = 0, flushed = 0;
  int r_len = 0;                 // run ordinal = lane (mod 32): its length ...
  unsigned long long r_dst = 0;  // ... and its table row
  float acc[4 * SS::kQuads];
  while (ok) {
    unsigned q = 0;
    if (lane == 0) q = atomicAdd(&p.work[1], 1u);
    q = __shfl_sync(kFull, q, 0);
    if (q >= n_st) break;
    const long long gi = q / ncb;
    const long long c0 = ((long long)q - gi * ncb) * kShortCols;
    const long long s1 = p.gstart[gi + 1];
    long long ps = p.gstart[gi];
    Window<int> sw;
    sw.init(p.seg, total + 1, ps, lane);
    Window<unsigned long long> pw;
    pw.init(p.rtab, total, ps, lane);
    Window<int> kw;
    kw.init(p.rows, nkeys, sw.at(ps, lane), lane);
    long long pk = 0, pend = 0;
    bool pdone = false;
    // keeps the ring full: the rows of the task's short runs in order, a
    // run's table slice issued with its first row
    auto top_up = [&]() {
      while (!pdone && issued - consumed < unsigned(C::kRS)) {
        if (pk == pend) {
          int a = 0, b = 0;
          for (;;) {
            if (ps >= s1) {
              pdone = true;
              break;
            }
            sw.pair(ps, lane, a, b);
            if (b - a <= kHeavyRows) break;
            ++ps;  // a long run: its CTA tasks sum it
          }
          if (pdone || run_ord - flushed >= unsigned(kTRing)) break;
          const unsigned long long tp = pw.at(ps, lane);
          const float* trow = reinterpret_cast<const float*>(tp);
          const int ts = int(run_ord % kTRing);
#pragma unroll
          for (int qd = 0; qd < SS::kQuads; ++qd) {
            const long long col = SS::quad_col(c0, lane, qd);
            cp_async16(&sm.table[w][ts][qd][lane], col < h ? trow + col : trow, col < h ? 16u : 0u);
          }
          if (lane == int(run_ord & 31u)) {
            r_len = b - a;
            r_dst = tp;
          }
          ++run_ord;
          ++ps;
          pk = a;
          pend = b;
        }
        const int row = kw.at(pk, lane);
        const int slot = int(issued % C::kRS);
        stage_row<EB, kShortCols>(ring, slot, lane, p.grad + (long long)row * p.ld_grad_bytes, c0, h,
                                  &sm.bar_s[w][slot]);
        ++issued;
        ++pk;
      }
    };
    top_up();
    while (ok && consumed < issued) {
      const int ts = int(flushed % kTRing);
      const int len = __shfl_sync(kFull, r_len, int(flushed & 31u));
      float* trow = reinterpret_cast<float*>(__shfl_sync(kFull, r_dst, int(flushed & 31u)));
#pragma unroll
      for (int e = 0; e < 4 * SS::kQuads; ++e) acc[e] = 0.f;
      for (int r = 0; r < len; ++r) {
        const int slot = int(consumed % C::kRS);
        ok = mbar_wait_warp(&sm.bar_s[w][slot], (consumed / C::kRS) & 1u);
        if (!ok) break;
        add_row<EB, kShortCols>(ring, slot, lane, acc);
        ++consumed;
        top_up();
      }
      if (!ok) break;
      // the table slice arrived with the run's first row
#pragma unroll
      for (int qd = 0; qd < SS::kQuads; ++qd) {
        const long long col = SS::quad_col(c0, lane, qd);
        if (col >= h) continue;
        float4 o = sm.table[w][ts][qd][lane];
        o.x += acc[4 * qd + 0];
        o.y += acc[4 * qd + 1];
        o.z += acc[4 * qd + 2];
        o.w += acc[4 * qd + 3];
        *reinterpret_cast<float4*>(trow + col) = o;
      }
      ++flushed;
      top_up();
    }
  }
  if (!ok && lane == 0) atomicOr(&p.hdr->error_flag, VPCE_FLAG_WAIT_TIMEOUT);
  cp_async_wait_all();  // nothing lands in shared memory after the CTA ends
}

int g_accum_ctas[2] = {1, 1};  // resident CTAs per SM of embed_accum_kernel<2>, <4>

}  // namespace

// Workspace: a header (its error flag is where vpce_read_error_flag looks),
// the sorted keys, the run starts, the long-run list, the group starts, the
// runs' table rows and the counters.
struct EmbedWs {
  Header* hdr;
  int* rows;
  int* seg;
  int* heavy;
  int* gstart;
  unsigned long long* rtab;
  int* counts;  // n_seg, n_heavy, n_grp, work[2]
};

size_t embed_bwd_workspace_bytes() {
  return 256 + round256(sizeof(int) * kEmbChunk) + round256(sizeof(int) * (kEmbChunk + 1)) +
         round256(sizeof(int) * (kEmbChunk / kHeavyRows)) + round256(sizeof(int) * (kEmbChunk / kGroupRows + 1)) +
         round256(sizeof(unsigned long long) * kEmbChunk) + 256;
}

EmbedWs embed_ws(void* ws) {
  unsigned char* w = static_cast<unsigned char*>(ws);
  EmbedWs e;
  e.hdr = reinterpret_cast<Header*>(w);
  w += 256;
  e.rows = reinterpret_cast<int*>(w);
  w += round256(sizeof(int) * kEmbChunk);
  e.seg = reinterpret_cast<int*>(w);
  w += round256(sizeof(int) * (kEmbChunk + 1));
  e.heavy = reinterpret_cast<int*>(w);
  w += round256(sizeof(int) * (kEmbChunk / kHeavyRows));
  e.gstart = reinterpret_cast<int*>(w);
  w += round256(sizeof(int) * (kEmbChunk / kGroupRows + 1));
  e.rtab = reinterpret_cast<unsigned long long*>(w);
  w += round256(sizeof(unsigned long long) * kEmbChunk);
  e.counts = reinterpret_cast<int*>(w);
  return e;
}

// keys of all blocks plus the CTA's sorted slice
size_t sort_smem_bytes(int n_pow2, size_t key_bytes) { return size_t(kSortCtas + 1) * (n_pow2 / kSortCtas) * key_bytes; }

cudaError_t set_embed_smem() {
  cudaError_t e = cudaFuncSetAttribute(embed_sort_runs_kernel<unsigned>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       int(sort_smem_bytes(kEmbChunk, 4)));
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(embed_sort_runs_kernel<unsigned long long>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             int(sort_smem_bytes(kEmbChunk, 8)));
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(embed_accum_kernel<2>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             int(sizeof(AccSmem<2>)));
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(embed_accum_kernel<4>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             int(sizeof(AccSmem<4>)));
  if (e == cudaSuccess)
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&g_accum_ctas[0], embed_accum_kernel<2>, kAThreads,
                                                      sizeof(AccSmem<2>));
  if (e == cudaSuccess)
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&g_accum_ctas[1], embed_accum_kernel<4>, kAThreads,
                                                      sizeof(AccSmem<4>));
  for (int& c : g_accum_ctas) c = c < 1 ? 1 : c;
  return e;
}

void launch_embed_forward(const ShardSet& sh, int t, long long V, long long h, int eb, const long long* ids,
                          long long s, void* out, long long ld_out, int* flag, int sms, cudaStream_t st) {
  EmbedFwdParams p;
  p.sh = sh;
  p.t = t;
  p.V = V;
  p.h = h;
  p.eb = eb;
  p.ids = ids;
  p.s = s;
  p.out = static_cast<unsigned char*>(out);
  p.ld_out_bytes = ld_out * eb;
  p.flag = flag;
  const long long want = (s + kEmbThreads / 32 - 1) / (kEmbThreads / 32);
  const long long cap = (long long)sms * 8;
  embed_forward_kernel<<<int(want < cap ? want : cap), kEmbThreads, 0, st>>>(p);
}

// Chunk after chunk: sort, then accumulate.  Returns the last launch error.
cudaError_t launch_embed_backward(const void* grad, int grad_bf16, long long ld_grad, const long long* ids,
                                  long long s, const ShardSet& gsh, int t, long long V, long long h, void* ws,
                                  int sms, cudaStream_t st) {
  const EmbedWs W = embed_ws(ws);
  int* n_seg = W.counts;
  int* n_heavy = W.counts + 1;
  int* n_grp = W.counts + 2;
  unsigned* work = reinterpret_cast<unsigned*>(W.counts + 3);
  const int eb = grad_bf16 ? 2 : 4;
  for (long long r0 = 0; r0 < s; r0 += kEmbChunk) {
    const int n = int(s - r0 < kEmbChunk ? s - r0 : kEmbChunk);
    int n2 = kSortCtas;
    while (n2 < n) n2 <<= 1;
    EmbedSortParams sp;
    sp.ids = ids + r0;
    sp.n = n;
    sp.n_pow2 = n2;
    sp.V = V;
    sp.rows = W.rows;
    sp.seg = W.seg;
    sp.heavy = W.heavy;
    sp.gstart = W.gstart;
    sp.rtab = W.rtab;
    sp.counts = W.counts;
    sp.hdr = W.hdr;
    sp.first = r0 == 0;
    sp.gsh = gsh;
    sp.t = t;
    if (V <= kMaxV32)
      embed_sort_runs_kernel<unsigned><<<kSortCtas, kSortThreads, sort_smem_bytes(n2, 4), st>>>(sp);
    else
      embed_sort_runs_kernel<unsigned long long><<<kSortCtas, kSortThreads, sort_smem_bytes(n2, 8), st>>>(sp);
    EmbedAccParams ap;
    ap.rows = W.rows;
    ap.seg = W.seg;
    ap.n_seg = n_seg;
    ap.heavy = W.heavy;
    ap.n_heavy = n_heavy;
    ap.grad = static_cast<const unsigned char*>(grad) + r0 * ld_grad * eb;
    ap.ld_grad_bytes = ld_grad * eb;
    ap.grad_bf16 = grad_bf16;
    ap.h = h;
    ap.gsh = gsh;
    ap.t = t;
    ap.gstart = W.gstart;
    ap.n_grp = n_grp;
    ap.rtab = W.rtab;
    ap.work = work;
    ap.hdr = W.hdr;
    // persistent: as many CTAs as fit take tasks until both lists are done
    if (grad_bf16)
      embed_accum_kernel<2><<<sms * g_accum_ctas[0], kAThreads, sizeof(AccSmem<2>), st>>>(ap);
    else
      embed_accum_kernel<4><<<sms * g_accum_ctas[1], kAThreads, sizeof(AccSmem<4>), st>>>(ap);
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

}  // namespace vpce
