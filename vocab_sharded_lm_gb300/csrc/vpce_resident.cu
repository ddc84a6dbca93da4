// Fused forward + backward with every row resident on chip: the logits cross
// HBM exactly once in each direction.
//
// The method ("Distributed Training III: Model Parallelism", CMU 11-868
// Lecture 16 notes, §5.5; "LLM Internals" §7.3.4) splits a row of logits over
// t vocabulary shards; each shard reduces its maximum, its sum of exponentials
// and, where it holds it, the target logit, and the three scalars combine into
// logsumexp - target.  Here a row is split over the C CTAs of a thread-block
// cluster instead (C = 1 when a row fits one CTA): each CTA owns a fixed byte
// range of every row ("its part", made of whole 16-byte chunks of the shard
// segments) and keeps the part of the current row in shared memory.
//
// Each of the 8 warps of a CTA owns a contiguous 1/8 of the CTA's part and a
// ring of six 4 KB shared-memory slots, and streams its own chunks of
// successive rows into that ring (cp.async.bulk, mbarrier per slot) up to six
// chunks ahead:
//                   pass 1: (max, sum-exp) over the warp's chunks of the row;
//                   the CTA merges its warps in order, then every CTA sends
//                   (M, S, target logit) to every CTA of the cluster through
//                   distributed shared memory -- the on-chip stand-in for the
//                   pages' max / sum / target all-reduces -- and folds the C
//                   entries in rank order, so all CTAs hold the same lse;
//                   pass 2: dlogits computed in the still-resident chunks and
//                   written over the logits by cp.async.bulk stores; a slot is
//                   refilled with a later chunk once its store has read it.
//   Pass 1 of the next row runs before pass 2 of the current one, so the
//   cluster exchange of a row overlaps useful work.
//
// Waits on mbarriers are bounded (about a second); the two cluster barriers
// (after set-up, before exit) are reached by every thread in bounded time.
#include "vpce_chunk.cuh"

namespace vpce {

namespace {

constexpr int kResWarps = 16;
constexpr int kResThreads = kResWarps * 32;
constexpr int kResChunk = 4096;
constexpr int kResSlots = 3;          // ring slots per warp
constexpr int kResMaxPerWarp = 4;     // chunk-table entries per warp
constexpr int kResMaxCluster = 8;
constexpr int kResMail = 4;           // mailbox buffers (rows in flight across the cluster)
constexpr int kResVPL = kResChunk / 512;

struct ResParams {
  ShardSet sh;
  int t;
  long long s;
  long long V;
  const long long* targets;
  long long ignore_index;
  int reduction;
  float grad;
  float* lse;
  float* rowl;
  float* row_loss;
  float* loss_out;
  Header* hdr;
};

struct ResSmem {
  unsigned char ring[kResWarps][kResSlots][kResChunk];
  uint64_t full[kResWarps][kResSlots];
  uint64_t mailbar[kResMail];
  unsigned arrived[2];                    // warps done with pass 1 of a row
  float4 mail[kResMail][kResMaxCluster];  // (M, S, target logit, holds target) per CTA rank
  float2 cpart[2][kResWarps];             // per warp (m, sum-exp)
  float tz[2];
  int cnt[kResWarps];
  int seg[kResWarps][kResMaxPerWarp];
  unsigned off[kResWarps][kResMaxPerWarp];
  unsigned len[kResWarps][kResMaxPerWarp];
};

}  // namespace

// Chunks of warp `w` of CTA `c` in a cluster of C, for rows made of t shard
// segments (widths in bytes are 16-byte multiples): the CTA's part is bytes
// [lo, hi) of the row, the warp's share is a contiguous 1/8 of it, cut at
// segment boundaries and into near-equal 16-byte aligned pieces of at most
// kResChunk.  Writes up to `cap` entries; returns the count.
__host__ __device__ inline int resident_chunks(const long long* start, int t, int eb, int C, int c, int w, int cap,
                                               int* seg, unsigned* off, unsigned* len) {
  unsigned long long R = 0;
  for (int i = 0; i < t; ++i) R += (unsigned long long)(start[i + 1] - start[i]) * eb;
  const unsigned long long plo = (R * c / C) & ~15ull;
  const unsigned long long phi = c == C - 1 ? R : (R * (c + 1) / C) & ~15ull;
  const unsigned long long lo = plo + (((phi - plo) * w / kResWarps) & ~15ull);
  const unsigned long long hi = w == kResWarps - 1 ? phi : plo + (((phi - plo) * (w + 1) / kResWarps) & ~15ull);
  unsigned long long pos = 0;
  int n = 0;
  for (int i = 0; i < t; ++i) {
    const unsigned long long W = (unsigned long long)(start[i + 1] - start[i]) * eb;
    const unsigned long long a0 = lo > pos ? lo : pos;
    const unsigned long long b0 = hi < pos + W ? hi : pos + W;
    if (a0 < b0) {
      const unsigned a = unsigned(a0 - pos), b = unsigned(b0 - pos);
      const unsigned nk = (b - a + kResChunk - 1) / kResChunk;
      for (unsigned k = 0; k < nk; ++k) {
        const unsigned ca = a + (unsigned((unsigned long long)(b - a) * k / nk) & ~15u);
        const unsigned cb = k + 1 == nk ? b : a + (unsigned((unsigned long long)(b - a) * (k + 1) / nk) & ~15u);
        if (n < cap && seg != nullptr) {
          seg[n] = i;
          off[n] = ca;
          len[n] = cb - ca;
        }
        ++n;
      }
    }
    pos += W;
  }
  return n;
}

namespace {

template <typename T>
__global__ void __launch_bounds__(kResThreads, 1) resident_kernel(const __grid_constant__ ResParams p) {
  constexpr int EB = Elem<T>::kBytes;
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  ResSmem& sm = *reinterpret_cast<ResSmem*>(smem_raw);
  __shared__ bool last;
  __shared__ double sv[kResWarps];
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t C = cluster_size();
  const uint32_t crank = cluster_rank();
  const long long q = cluster_id();
  const long long nq = cluster_count();

  if (lane == 0) {
    sm.cnt[warp] = resident_chunks(p.sh.start, p.t, EB, int(C), int(crank), warp, kResMaxPerWarp, sm.seg[warp],
                                   sm.off[warp], sm.len[warp]);
    for (int k = 0; k < kResSlots; ++k) mbar_init(&sm.full[warp][k], 1);
    if (warp == 0) {
      sm.arrived[0] = 0u;
      sm.arrived[1] = 0u;
      for (int b = 0; b < kResMail; ++b) mbar_init(&sm.mailbar[b], C);
    }
    fence_mbar_init();
  }
  __syncthreads();
  cluster_sync_all();  // peers' barriers exist before any remote arrive

  const int cw = sm.cnt[warp];
  const int* seg = sm.seg[warp];
  const unsigned* off = sm.off[warp];
  const unsigned* len = sm.len[warp];
  const int n_valid = p.hdr->n_valid;
  const float scale = p.reduction == VPCE_SUM ? p.grad : (n_valid > 0 ? p.grad / float(n_valid) : 0.f);
  bool alive = true;
  for (int w = 0; w < kResWarps; ++w)
    alive = alive && sm.cnt[w] <= kResMaxPerWarp && 2 * sm.cnt[w] <= kResSlots;
  const uint64_t pol = policy_evict_first();

  // ---- loads: this warp's chunks of successive non-ignored rows, in order;
  // chunk i goes to slot i % kResSlots
  long long pr = q;  // row of the next chunk to load
  int pj = 0;        // its index in the warp's table
  unsigned issued = 0;
  auto seek_row = [&](long long from) {
    pr = from;
    while (pr < p.s && __ldg(p.targets + pr) == p.ignore_index) pr += nq;
  };
  auto issue_next = [&]() {
    if (cw == 0 || pr >= p.s) return;
    const int slot = int(issued % kResSlots);
    if (lane == 0) {
      const int i = seg[pj];
      mbar_arrive_expect_tx(&sm.full[warp][slot], len[pj]);
      bulk_load(sm.ring[warp][slot], p.sh.ptr[i] + pr * p.sh.ld_bytes[i] + off[pj], len[pj],
                &sm.full[warp][slot], pol);
    }
    ++issued;
    if (++pj == cw) {
      pj = 0;
      seek_row(pr + nq);
    }
  };
  if (alive) {
    seek_row(q);
    for (int k = 0; k < kResSlots; ++k) issue_next();
  }

  // next row to process; ignored rows met on the way get zeros over this
  // warp's share (nothing is read)
  auto next_row = [&](long long from) -> long long {
    for (long long r = from; r < p.s; r += nq) {
      if (__ldg(p.targets + r) != p.ignore_index) return r;
      for (int j = 0; j < cw; ++j) {
        uint4* d = reinterpret_cast<uint4*>(const_cast<unsigned char*>(p.sh.ptr[seg[j]]) +
                                            r * p.sh.ld_bytes[seg[j]] + off[j]);
        for (unsigned v = lane; v < (len[j] >> 4); v += 32) d[v] = make_uint4(0u, 0u, 0u, 0u);
      }
      if (crank == 0 && warp == 0 && lane == 0) {
        p.rowl[r] = 0.f;
        p.lse[r] = 0.f;
        if (p.row_loss) p.row_loss[r] = 0.f;
      }
    }
    return p.s;
  };
  // segment and byte offset of row r's target (segment -1: none in range)
  auto target_of = [&](long long y, int& ty, unsigned& toff) {
    ty = -1;
    toff = 0;
    if (y >= 0 && y < p.V) {
      ty = 0;
      while (p.sh.start[ty + 1] <= y) ++ty;
      toff = unsigned(y - p.sh.start[ty]) * EB;
    }
  };
  // pass 1 of the n-th processed row r; the CTA's partial goes to every CTA
  // of the cluster
  auto pass1 = [&](long long r, unsigned n) -> bool {
    int ty;
    unsigned toff;
    target_of(__ldg(p.targets + r), ty, toff);
    const int buf = int(n & 1u);
    float m = -INFINITY, se = 0.f;
#pragma unroll 1
    for (int j = 0; j < cw; ++j) {
      const unsigned i = n * unsigned(cw) + unsigned(j);
      const int slot = int(i % kResSlots);
      if (!mbar_wait_warp(&sm.full[warp][slot], (i / kResSlots) & 1u)) return false;
      stats_chunk<kResVPL>(sm.ring[warp][slot], len[j], lane, m, se, T());
      if (lane == 0 && seg[j] == ty && toff >= off[j] && toff < off[j] + len[j])
        sm.tz[buf] = Elem<T>::load(sm.ring[warp][slot] + (toff - off[j]));
    }
    warp_merge_ms(m, se);
    // the last warp of the CTA to finish the row merges every warp's partial
    // (in warp order) and sends the CTA's (M, S, target) to the cluster;
    // nobody waits here
    bool last_warp = false;
    if (lane == 0) {
      sm.cpart[buf][warp] = make_float2(m, se);
      __threadfence_block();
      last_warp = atomicAdd(&sm.arrived[buf], 1u) == unsigned(kResWarps - 1);
    }
    last_warp = __shfl_sync(kFull, last_warp, 0);
    if (last_warp) {
      __threadfence_block();
      float M = sm.cpart[buf][0].x, S = sm.cpart[buf][0].y;
#pragma unroll
      for (int w = 1; w < kResWarps; ++w) merge_ms(M, S, sm.cpart[buf][w].x, sm.cpart[buf][w].y);
      bool mine = false;
      if (lane < kResWarps) {
        const int cnt = sm.cnt[lane];
        for (int j = 0; j < cnt; ++j)
          mine |= sm.seg[lane][j] == ty && toff >= sm.off[lane][j] && toff < sm.off[lane][j] + sm.len[lane][j];
      }
      mine = __any_sync(kFull, mine);
      const float zt = mine ? sm.tz[buf] : 0.f;
      if (lane == 0) sm.arrived[buf] = 0u;  // reused two rows later, after the cluster exchange
      const int mb = int(n % kResMail);
      if (lane < int(C)) {
        st_cluster_v4(map_to_rank(smem_addr(&sm.mail[mb][crank]), uint32_t(lane)), M, S, zt, mine ? 1.f : 0.f);
        mbar_arrive_cluster(map_to_rank(smem_addr(&sm.mailbar[mb]), uint32_t(lane)));
      }
    }
    return true;
  };
  // the cluster-wide lse of the n-th row r, then pass 2: dlogits in the
  // resident chunks, bulk-stored over the logits; each slot is refilled with
  // the chunk kResSlots further on once its store has read it
  auto pass2 = [&](long long r, unsigned n) -> bool {
    const long long y = __ldg(p.targets + r);
    int ty;
    unsigned toff;
    target_of(y, ty, toff);
    const int mb = int(n % kResMail);
    if (!mbar_wait_warp_cluster(&sm.mailbar[mb], (n / kResMail) & 1u)) return false;
    float M = sm.mail[mb][0].x, S = sm.mail[mb][0].y;
    float zt = sm.mail[mb][0].w > 0.f ? sm.mail[mb][0].z : 0.f;
    for (int j = 1; j < int(C); ++j) {
      const float4 e = sm.mail[mb][j];
      merge_ms(M, S, e.x, e.y);
      if (e.w > 0.f) zt = e.z;
    }
    const bool in_range = ty >= 0;
    const float lse = in_range ? M + logf(S) : __int_as_float(0x7fc00000);
    if (crank == 0 && warp == 0 && lane == 0) {
      const float rl = in_range ? lse - zt : lse;
      p.lse[r] = lse;
      p.rowl[r] = rl;
      if (p.row_loss) p.row_loss[r] = rl;
    }
    const float c = -lse * kLog2e;
#pragma unroll 1
    for (int j = 0; j < cw; ++j) {
      const unsigned i = n * unsigned(cw) + unsigned(j);
      const int slot = int(i % kResSlots);
      unsigned char* buf = sm.ring[warp][slot];
      const int tb = (seg[j] == ty && toff >= off[j] && toff < off[j] + len[j]) ? int(toff - off[j]) : -1;
      float dt = 0.f;
      if (tb >= 0 && lane == 0) dt = (ex2(fmaf(Elem<T>::load(buf + tb), kLog2e, c)) - 1.f) * scale;
      __syncwarp();
      grad_chunk<T, kResVPL>(buf, len[j], lane, c, scale);
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
        if (tb >= 0) {
          Elem<T>::store(buf + tb, dt);
          fence_proxy_async_smem();
        }
        bulk_store(const_cast<unsigned char*>(p.sh.ptr[seg[j]]) + r * p.sh.ld_bytes[seg[j]] + off[j], buf, len[j],
                   pol);
        bulk_commit();
      }
      if (j > 0) {
        if (lane == 0) bulk_wait_read<1>();
        __syncwarp();
        issue_next();  // refills the slot of chunk i - 1
      }
    }
    if (cw > 0) {
      if (lane == 0) bulk_wait_read<0>();
      __syncwarp();
      issue_next();  // refills the slot of the row's last chunk
    }
    return true;
  };

  if (alive) {
    unsigned n = 0;
    long long r = next_row(q);
    if (r < p.s) alive = pass1(r, 0);
    while (alive && r < p.s) {
      const long long rn = next_row(r + nq);
      if (rn < p.s && !pass1(rn, n + 1)) {
        alive = false;
        break;
      }
      if (!pass2(r, n)) {
        alive = false;
        break;
      }
      r = rn;
      ++n;
    }
  }
  if (!alive) {
    if (lane == 0) atomicOr(&p.hdr->error_flag, VPCE_FLAG_WAIT_TIMEOUT);
    // the latest load of every slot lands before this warp's shared memory is
    // released
    for (unsigned i = issued > unsigned(kResSlots) ? issued - kResSlots : 0u; i < issued; ++i)
      if (!mbar_wait_warp(&sm.full[warp][i % kResSlots], (i / kResSlots) & 1u)) break;
  }
  if (lane == 0) bulk_wait_all<0>();  // every dlogits store has landed

  __syncthreads();
  cluster_sync_all();  // no CTA leaves while a peer may still touch its shared memory

  // ---- batch loss: the last block sums the per-row losses in a fixed order
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) last = atomicAdd(&p.hdr->ticket, 1u) == gridDim.x - 1;
  __syncthreads();
  if (!last) return;
  __threadfence();
  double v = 0.0;
  const long long nb = (p.s + 255) / 256;
  for (long long b = threadIdx.x; b < nb; b += kResThreads) {
    double bs = 0.0;
    const long long e = min(p.s, (b + 1) * 256);
    for (long long r = b * 256; r < e; ++r) bs += double(__ldcg(p.rowl + r));
    v += bs;
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_down_sync(kFull, v, o);
  if (lane == 0) sv[warp] = v;
  __syncthreads();
  if (threadIdx.x == 0) {
    double tot = 0.0;
    for (int i = 0; i < kResWarps; ++i) tot += sv[i];
    const int cnt = p.hdr->n_valid;
    p.hdr->loss_sum = tot;
    p.hdr->ticket = 0u;
    *p.loss_out =
        p.reduction == VPCE_SUM ? float(tot) : (cnt > 0 ? float(tot / double(cnt)) : __int_as_float(0x7fc00000));
  }
}

struct ResLaunchCache {
  int clusters[kResMaxCluster + 1][2];  // [C][bf16] co-resident clusters, 0 = unknown, -1 = none
};
ResLaunchCache g_res_cache[64];

}  // namespace

cudaError_t set_resident_smem() {
  cudaError_t e = cudaFuncSetAttribute(resident_kernel<float>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       int(sizeof(ResSmem)));
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(resident_kernel<__nv_bfloat16>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              int(sizeof(ResSmem)));
}

// Cluster size for the resident kernel.  A warp's share of a row must fit its
// ring twice (pass 1 of the next row runs before pass 2 of the current one
// frees the slots); three times leaves room to stream a third row.  The
// smallest C (<= 8) whose shares fit three times, else 8 if they fit twice,
// else 0 (rows too long: the L2-reuse kernel runs instead).
int resident_cluster_size(const ShardSet& sh, int t, int eb) {
  auto worst = [&](int C) {
    int m = 0;
    for (int c = 0; c < C; ++c)
      for (int w = 0; w < kResWarps; ++w) {
        const int n = resident_chunks(sh.start, t, eb, C, c, w, 0, nullptr, nullptr, nullptr);
        m = n > m ? n : m;
      }
    return m;
  };
  for (int C = 1; C <= kResMaxCluster; ++C) {
    const int n = worst(C);
    if (n <= kResMaxPerWarp && 3 * n <= kResSlots) return C;
  }
  const int n8 = worst(kResMaxCluster);
  return (n8 <= kResMaxPerWarp && 2 * n8 <= kResSlots) ? kResMaxCluster : 0;
}

// Co-resident clusters of size C for the resident kernel on device `dev`
// (cached; -1 when none fits).
int resident_max_clusters(bool bf16, int C, int dev) {
  int& cached = g_res_cache[dev & 63].clusters[C][bf16 ? 1 : 0];
  if (cached == 0) {
    void* fn = bf16 ? reinterpret_cast<void*>(resident_kernel<__nv_bfloat16>)
                    : reinterpret_cast<void*>(resident_kernel<float>);
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = unsigned(C);
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.gridDim = dim3(unsigned(C) * 1024u, 1, 1);
    cfg.blockDim = dim3(kResThreads, 1, 1);
    cfg.dynamicSmemBytes = sizeof(ResSmem);
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, fn, &cfg) != cudaSuccess || n <= 0) {
      cudaGetLastError();
      cached = -1;
    } else {
      cached = n;
    }
  }
  return cached;
}

// Launch the resident kernel with clusters of C; returns false (nothing
// launched) when no cluster of that size can be resident.
bool launch_resident(const ShardSet& sh, bool bf16, int C, int t, long long s, long long V, const long long* targets,
                     long long ignore_index, int reduction, float grad, float* lse, float* rowl, float* row_loss,
                     float* loss_out, Header* hdr, int dev, cudaStream_t st) {
  ResParams p;
  p.sh = sh;
  p.t = t;
  p.s = s;
  p.V = V;
  p.targets = targets;
  p.ignore_index = ignore_index;
  p.reduction = reduction;
  p.grad = grad;
  p.lse = lse;
  p.rowl = rowl;
  p.row_loss = row_loss;
  p.loss_out = loss_out;
  p.hdr = hdr;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = unsigned(C);
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.blockDim = dim3(kResThreads, 1, 1);
  cfg.dynamicSmemBytes = sizeof(ResSmem);
  cfg.stream = st;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const int cached = resident_max_clusters(bf16, C, dev);
  if (cached < 0) return false;
  long long clusters = cached;
  if (clusters > s) clusters = s;
  cfg.gridDim = dim3(unsigned(clusters * C), 1, 1);
  if (bf16) cudaLaunchKernelEx(&cfg, resident_kernel<__nv_bfloat16>, p);
  else cudaLaunchKernelEx(&cfg, resident_kernel<float>, p);
  return true;
}

}  // namespace vpce
