// Fused forward + backward of the vocab-parallel cross-entropy for rows of
// any length: the loss and the in-place dlogits with the logits read from HBM
// once, re-read from L2 and written once.
//
// The method ("Distributed Training III: Model Parallelism", CMU 11-868
// Lecture 16 notes, §5.5; "LLM Internals" §7.3.4) reduces per row the maximum,
// the sum of exponentials and the target logit over the vocabulary shards and
// combines them into logsumexp - target.  When the upstream gradient g is known
// up front (the loss is the last op, g = 1 or a loss scale), the backward of a
// row can follow its forward while the row is still on chip:
//
//   * a CTA owns whole rows; its 8 "stats" warps each take 1/8 of a row (one
//     contiguous range of its shard segments) and stream it from HBM through their own shared-memory
//     rings (cp.async.bulk + mbarrier), keeping an online (max, sum-exp) --
//     the streaming pattern of the split forward;
//   * per row they leave 8 partials (and the target logit) in a two-deep
//     shared-memory mailbox -- the on-chip stand-in for the pages' max / sum /
//     target all-reduces (rows over 224 KB are shared by a cluster of two
//     CTAs, which also send their partials to each other's mailboxes);
//   * 8 "grad" warps follow about a row behind: they fold the partials in warp
//     order into logsumexp, re-read the same bytes (L2 hits: the stats warps
//     fetched them microseconds earlier), turn them into dlogits in shared
//     memory and write them over the logits with cp.async.bulk stores -- the
//     pattern of the split backward.
//
// HBM sees one read and one write of the logits.  The batch count n_valid
// (needed for the 1/n_valid of the mean before any gradient is written) comes
// from a one-block prologue kernel that also clears the workspace header; the
// batch loss is summed in a fixed order by the last block to finish.
#include <mutex>

#include "vpce_chunk.cuh"

namespace vpce {

namespace {

constexpr int kPrepThreads = 1024;

// The fused kernel is the prologue's programmatic dependent (see
// grid_dependency_wait): it may start while the prologue still runs, and
// only its grad warps, and every thread before the batch-loss ticket, wait
// for it.  Measured on GB300: 0.7129 -> 0.7071 ms per call at s = 8192.
constexpr int kSW = 8;         // stats warps
constexpr int kSWLog2 = 3;
constexpr int kDW = 8;         // grad warps
constexpr int kFThreads = (kSW + kDW) * 32;
constexpr int kFChunk = 4096;  // bytes per pipeline chunk
// Ring slots per stats warp (HBM latency) and per grad warp (L2 latency, and
// the slot its last store still reads).  Measured on GB300 with the same
// 224 KB of rings: 3 and 4 beat 4 and 3 by 1.2% at s = 8192 (bf16, one CTA
// per row) and by 4.6% at s = 16384 (fp32, CTA pairs); 5 and 2 lose 14%.
constexpr int kSSlots = 3;
constexpr int kDSlots = 4;
// L2 bytes per CTA the two passes may keep live between them: one row is
// the least (a row's statistics precede its gradient); rows shorter than
// this let the stats warps run further ahead.  Measured on GB300 with each
// warp taking one contiguous range of the row and one CTA per row: 288 KB
// per SM (44 MB over 152 SMs; one 4 KB chunk of slack per stats warp for
// 250 KB rows) gave 0.664 ms at s = 8192, V = 128256, against 0.685 ms with
// 320 KB (two chunks), 0.753 ms with 352 KB and 0.715 ms with no slack;
// 100 KB rows (s = 4096) run the same with 288, 320 or 352 KB.
constexpr unsigned kLiveBytesPerCta = 288u * 1024u;
// Rows longer than this are shared by a pair of CTAs; shorter ones run on
// one CTA, with whatever slack the window above leaves.  Measured on GB300:
// s = 8192, V = 128256 (250 KB rows) 0.660 ms on one CTA per row against
// 0.654 ms on pairs (125 KB half rows, five chunks of slack); s = 4096,
// V = 50304 (98 KB rows) 0.167 ms against 0.206 ms.
constexpr long long kPairRowBytes = 224ll * 1024ll;
// The same budget for CTAs that share rows (a cluster per row): their row
// statistics also cross SMs.  Measured on GB300: s = 32768 bf16 (half rows
// of 250 KB) 5.16 ms with 288 KB (one chunk of slack per stats warp),
// 5.34 ms with 320 KB, 5.69 ms with 256 or 352 KB; s = 8192 (125 KB half
// rows) 0.654 ms, within 0.3% of 224 and 256 KB, 0.672 ms with 320 KB;
// s = 16384 fp32 (304 KB half rows, no slack) the same with 256, 288 or
// 320 KB.
constexpr unsigned kLiveBytesPerCtaShared = 288u * 1024u;
// stats warp w and grad warp w walk the same chunks: the credit between them
// counts those chunks
static_assert(kSW == kDW, "stats and grad warps pair up");
static_assert((1 << kSWLog2) == kSW, "a row part's warp count is a power of two");
constexpr int kFVPL = kFChunk / 512;

struct FusedParams {
  ShardSet sh;
  int t;
  long long s;
  long long V;
  const long long* targets;
  long long ignore_index;
  int reduction;
  float grad;
  unsigned credit_slack;   // chunks a stats warp may run past one row ahead of its grad partner
  const float* grad_rows;  // [s] per-row upstream gradient, or null (use grad)
  float* lse;       // [s]
  float* rowl;      // [s]: per-row loss (0 ignored, NaN bad target)
  float* row_loss;  // optional user copy of rowl
  float* loss_out;  // may be null ('none')
  Header* hdr;
};

// The shard geometry, copied from the kernel parameters into shared memory
// once per CTA: the chunk walk looks a segment up several times per chunk,
// and a run-time index into the parameter block costs a dependent
// constant-cache load each time.
struct Geo {
  const unsigned char* ptr[VPCE_MAX_SHARDS];
  long long ld[VPCE_MAX_SHARDS];
  int start[VPCE_MAX_SHARDS + 1];  // V < 2^31
};

struct FusedSmem {
  unsigned char sring[kSW][kSSlots][kFChunk];
  unsigned char dring[kDW][kDSlots][kFChunk];
  uint64_t sfull[kSW][kSSlots];
  uint64_t dfull[kDW][kDSlots];
  uint64_t rowdone[2];  // stats warps -> grad warps: a row's partials are in
  uint64_t rowfree[2];  // grad warps -> stats warps: the grad warps have begun that row
  float2 part[2][2 * kSW];  // (max, sum exp) of every stats warp of the row's CTAs, CTA-rank major
  float tz[2];
  unsigned sdone[kSW];  // chunks stats warp w has received (its grad partner may re-read them)
  unsigned gdone[kDW];  // chunks grad warp w has received (credit back to its stats partner)
  Geo geo;
};
// Within the 227 KB of dynamic shared memory a CTA may use (the kernel has
// no static shared memory).
static_assert(sizeof(FusedSmem) <= 232448, "fused kernel shared memory");

// Prologue: clear the header, count the valid rows, flag bad targets.
__global__ void __launch_bounds__(kPrepThreads) prep_kernel(const long long* targets, long long s,
                                                            long long V, long long ignore_index, Header* hdr,
                                                            int reduction, float* loss_out) {
  // The header's error flag and ticket are cleared before the dependent fused
  // kernel may start, so that a bit it sets (a wait that gave up) is never
  // overwritten by this clear; the bad-target bit below is OR-ed in.
  if (threadIdx.x == 0) {
    hdr->error_flag = 0;
    hdr->ticket = 0u;
    __threadfence();
  }
  __syncthreads();
  grid_launch_dependents();  // the fused kernel's stats warps need nothing else from here
  __shared__ int sc[kPrepThreads / 32];
  __shared__ int sbad[kPrepThreads / 32];
  int c = 0, bad = 0;
  for (long long r = threadIdx.x; r < s; r += kPrepThreads) {
    const long long y = targets[r];
    if (y == ignore_index) continue;
    if (y < 0 || y >= V) bad = 1;
    else ++c;
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    c += __shfl_down_sync(kFull, c, o);
    bad |= __shfl_down_sync(kFull, bad, o);
  }
  if ((threadIdx.x & 31) == 0) {
    sc[threadIdx.x >> 5] = c;
    sbad[threadIdx.x >> 5] = bad;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    int tc = 0, tb = 0;
    for (int i = 0; i < kPrepThreads / 32; ++i) {
      tc += sc[i];
      tb |= sbad[i];
    }
    hdr->n_valid = tc;
    if (tb) atomicOr(&hdr->error_flag, VPCE_FLAG_BAD_TARGET);
    hdr->reduction = reduction;
    hdr->loss_sum = 0.0;
    if (s == 0 && loss_out != nullptr) *loss_out = reduction != VPCE_MEAN ? 0.f : __int_as_float(0x7fc00000);
  }
}

// The part of every row one warp of a role owns: the bytes [lo, hi) of the
// row's shard segments laid end to end (segment i starts at byte start[i] *
// element size), 16-byte aligned.  One CTA per row: the whole row, cut into
// kSW equal ranges.  A cluster of NR CTAs per row: with at least NR shards,
// CTA c takes the segments between the shard boundaries nearest c/NR and
// (c+1)/NR of the row (at least one each), with fewer shards the c-th NR-th
// of the row; its kSW warps then cut that part into equal ranges.  A range
// may cross segment boundaries, so a warp's chunks are full kFChunk bytes
// except where a segment or its range ends.
struct RowPart {
  int sa, sb;        // the segments the CTA's part touches
  unsigned lo, hi;   // this warp's bytes of the row
};

template <int NR, int EB>
__device__ __forceinline__ RowPart row_part(const Geo& g, int t, unsigned crank, int w) {
  RowPart rp{0, t, 0u, 0u};
  unsigned clo = 0, chi = unsigned(g.start[t]) * EB;
  if (NR > 1) {
    if (t < NR) {
      const unsigned long long len = chi;
      clo = unsigned((len * crank) / NR) & ~15u;
      chi = int(crank) == NR - 1 ? chi : unsigned((len * (crank + 1)) / NR) & ~15u;
    } else {
      int prev = 0;
      for (int c = 1; c <= int(crank) + 1; ++c) {
        int k = t;
        if (c < NR) {
          // the boundary nearest c/NR of the row, leaving a segment for each CTA
          long long best = -1;
          for (int i = prev + 1; i <= t - (NR - c); ++i) {
            const long long d = (long long)NR * g.start[i] - (long long)c * g.start[t];
            const long long ad = d < 0 ? -d : d;
            if (best < 0 || ad < best) {
              best = ad;
              k = i;
            }
          }
        }
        if (c == int(crank) + 1) {
          rp.sa = prev;
          rp.sb = k;
        }
        prev = k;
      }
      clo = unsigned(g.start[rp.sa]) * EB;
      chi = unsigned(g.start[rp.sb]) * EB;
    }
  }
  // kSW equal ranges of the CTA's part (a power of two: no division)
  const unsigned long long len = chi - clo;
  rp.lo = clo + (unsigned((len * unsigned(w)) >> kSWLog2) & ~15u);
  rp.hi = w == kSW - 1 ? chi : clo + (unsigned((len * unsigned(w + 1)) >> kSWLog2) & ~15u);
  // the segments the warp's range touches
  while (rp.sa + 1 < rp.sb && unsigned(g.start[rp.sa + 1]) * EB <= rp.lo) ++rp.sa;
  while (rp.sb - 1 > rp.sa && unsigned(g.start[rp.sb - 1]) * EB >= rp.hi) --rp.sb;
  return rp;
}

// Walks the chunks of row r in a warp's part: from lo to hi, kFChunk bytes
// at a time, a chunk ending early where a segment ends.  No division on the
// way: the walk runs once per chunk on the critical path of both roles,
// where a 64-bit division by a variable chunk count cost as much as the
// chunk's arithmetic.  bounds() gives a chunk's byte range inside its
// segment, addr() its address.
template <int EB>
struct RowWalk {
  int seg;
  unsigned pos, hi;     // the next chunk starts at row byte pos; the warp's range ends at hi
  unsigned seg_lo, seg_hi;  // row bytes of segment seg
  unsigned char* base;  // the row's first byte in shard seg
  bool ok;

  __device__ __forceinline__ void enter(const Geo& g, long long r) {
    seg_lo = unsigned(g.start[seg]) * EB;
    seg_hi = unsigned(g.start[seg + 1]) * EB;
    base = const_cast<unsigned char*>(g.ptr[seg]) + r * g.ld[seg];
  }
  __device__ __forceinline__ bool seek(const Geo& g, const RowPart& rp, long long r, int /*from*/) {
    pos = rp.lo;
    hi = rp.hi;
    seg = rp.sa;
    if (pos >= hi) return ok = false;
    while (unsigned(g.start[seg + 1]) * EB <= pos) ++seg;
    enter(g, r);
    return ok = true;
  }
  __device__ __forceinline__ void next(const Geo& g, const RowPart& /*rp*/, long long r) {
    pos = min(min(pos + unsigned(kFChunk), seg_hi), hi);
    if (pos >= hi) {
      ok = false;
      return;
    }
    if (pos >= seg_hi) {
      ++seg;
      enter(g, r);
    }
  }
  __device__ __forceinline__ void bounds(unsigned& a, unsigned& b) const {
    a = pos - seg_lo;
    b = min(min(pos + unsigned(kFChunk), seg_hi), hi) - seg_lo;
  }
  __device__ __forceinline__ unsigned char* addr(unsigned a) const { return base + a; }
};

// Chunks of one row in a warp's part (the same for every row).
template <int EB>
__device__ __forceinline__ unsigned row_chunks(const Geo& g, const RowPart& rp) {
  unsigned c = 0;
  for (int i = rp.sa; i < rp.sb; ++i) {
    const unsigned lo = max(rp.lo, unsigned(g.start[i]) * EB);
    const unsigned hi = min(rp.hi, unsigned(g.start[i + 1]) * EB);
    if (hi > lo) c += (hi - lo + kFChunk - 1) / kFChunk;
  }
  return c;
}

// The load side of a warp's walk: the chunks of its part of every row the
// CTA owns (rows r0, r0 + step, ...), ignored rows skipped, in the order the
// arithmetic consumes them.
template <int EB>
struct RowCursor {
  long long r, step;
  RowWalk<EB> wk;
  bool ok;

  __device__ __forceinline__ void start(const FusedParams& p, const Geo& g, const RowPart& rp, long long r0,
                                        long long st) {
    step = st;
    r = r0 - st;
    next_row(p, g, rp);
  }
  __device__ __forceinline__ void next_row(const FusedParams& p, const Geo& g, const RowPart& rp) {
    for (;;) {
      r += step;
      if (r >= p.s) {
        ok = false;
        return;
      }
      if (__ldg(p.targets + r) == p.ignore_index) continue;
      if (wk.seek(g, rp, r, 0)) {
        ok = true;
        return;
      }
    }
  }
  __device__ __forceinline__ void advance(const FusedParams& p, const Geo& g, const RowPart& rp) {
    wk.next(g, rp, r);
    if (!wk.ok) next_row(p, g, rp);
  }
};

__device__ __forceinline__ unsigned ld_volatile(const unsigned* a) { return *const_cast<const volatile unsigned*>(a); }
__device__ __forceinline__ void st_volatile(unsigned* a, unsigned v) { *const_cast<volatile unsigned*>(a) = v; }

// Bounded, warp-uniform wait until the shared counter *c (raised by another
// warp of the CTA) exceeds `floor`.
__device__ __forceinline__ bool wait_counter_above(const unsigned* c, unsigned floor) {
  if (__all_sync(kFull, ld_volatile(c) > floor)) return true;
  const long long t0 = clock64();
  for (;;) {
    __nanosleep(64);
    if (__all_sync(kFull, ld_volatile(c) > floor)) return true;
    if (__any_sync(kFull, clock64() - t0 > kWaitLimitCycles)) return false;
  }
}

// segment and byte offset of target y (segment -1 when out of range)
template <int EB>
__device__ __forceinline__ void target_of(const Geo& g, int t, long long y, int& ty, unsigned& toff) {
  ty = -1;
  toff = 0;
  if (y >= 0 && y < g.start[t]) {
    ty = 0;
    while (g.start[ty + 1] <= y) ++ty;
    toff = unsigned(y - g.start[ty]) * EB;
  }
}

// NR > 1: a cluster of NR CTAs shares each row, CTA c taking the c-th part
// of every warp role's column split (NR kSW stats warps per row).  Each CTA's
// live L2 window then holds part rows, which keeps rows longer than the
// live budget re-read from L2.  Each stats warp posts its partial to every
// CTA's mailbox: to its own with a store and an arrival on the row barrier
// (kSW arrivals), to the others with st.async, whose bytes the receiving
// barrier counts.  Every grad warp folds the NR kSW partials (one per lane,
// then a fixed butterfly), so all CTAs reach the same logsumexp.
template <typename T, int NR>
__global__ void __launch_bounds__(kFThreads, 1) stream_fused_kernel(const __grid_constant__ FusedParams p) {
  constexpr int EB = Elem<T>::kBytes;
  constexpr bool PAIR = NR > 1;     // CTAs of a cluster share each row
  static_assert(NR == 1 || NR == 2, "one row per CTA or per pair of CTAs");
  constexpr int NWR = NR * kSW;     // warps of one role per row
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  FusedSmem& sm = *reinterpret_cast<FusedSmem*>(smem_raw);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const bool stats = warp < kSW;
  const int w = stats ? warp : warp - kSW;
  const unsigned crank = PAIR ? cluster_rank() : 0u;

  if (lane == 0) {
    if (stats) {
      for (int k = 0; k < kSSlots; ++k) mbar_init(&sm.sfull[w][k], 1);
    } else {
      for (int k = 0; k < kDSlots; ++k) mbar_init(&sm.dfull[w][k], 1);
    }
    if (stats) sm.sdone[w] = 0u;
    else sm.gdone[w] = 0u;
    if (warp == 0) {
      mbar_init(&sm.rowdone[0], kSW);
      mbar_init(&sm.rowdone[1], kSW);
      mbar_init(&sm.rowfree[0], NR * kDW);
      mbar_init(&sm.rowfree[1], NR * kDW);
    }
    fence_mbar_init();
  }
  for (int i = threadIdx.x; i <= p.t; i += kFThreads) {
    sm.geo.start[i] = int(p.sh.start[i]);
    if (i < p.t) {
      sm.geo.ptr[i] = p.sh.ptr[i];
      sm.geo.ld[i] = p.sh.ld_bytes[i];
    }
  }
  __syncthreads();
  // the peer's barriers must be initialised before any arrival reaches them
  if (PAIR) cluster_sync_all();
  const Geo& geo = sm.geo;
  const int nt = p.t;
  const RowPart rp = row_part<NR, EB>(geo, nt, crank, w);  // this warp's part of every row
  // this CTA's bytes of a row (the union of its warps' ranges)
  const unsigned cta_lo = PAIR ? row_part<NR, EB>(geo, nt, crank, 0).lo : 0u;
  const unsigned cta_hi = PAIR ? row_part<NR, EB>(geo, nt, crank, kSW - 1).hi : 0u;

  const long long r_step = gridDim.x / NR;
  const long long r0 = blockIdx.x / NR;
  bool alive = true;
  auto wait_row_bar = [&](uint64_t* bar, uint32_t parity) {
    return PAIR ? mbar_wait_warp_cluster(bar, parity) : mbar_wait_warp(bar, parity);
  };

  if (stats) {
    // ---------------- stats warps: pass 1 from HBM.  The loads run ahead of
    // the arithmetic across row boundaries, limited by the ring and by the
    // credit from the grad partner: chunk i is loaded only once grad warp w
    // has received chunk i - budget, which keeps about one row per CTA (plus
    // the slack) live in L2 between the two passes.
    unsigned char(*ring)[kFChunk] = sm.sring[w];
    uint64_t* full = sm.sfull[w];
    // normal priority: the grad warps' loads and stores of these bytes are
    // marked evict-first, which frees their lines once re-read and rewritten
    // (on GB300 evict_last here measured 0.4% slower; dropping evict_first on
    // the grad side, 18% slower)
    const uint64_t pol = policy_evict_normal();
    const unsigned budget = row_chunks<EB>(geo, rp) + p.credit_slack;
    RowCursor<EB> prod;
    prod.start(p, geo, rp, r0, r_step);
    unsigned issued = 0, kc = 0, n = 0;
    auto top_up = [&]() {
      const unsigned credit = __shfl_sync(kFull, ld_volatile(&sm.gdone[w]), 0) + budget;
      while (prod.ok && issued < kc + kSSlots && issued < credit) {
        unsigned a, b;
        prod.wk.bounds(a, b);
        const int slot = int(issued % kSSlots);
        if (lane == 0) {
          mbar_arrive_expect_tx(&full[slot], b - a);
          bulk_load(ring[slot], prod.wk.addr(a), b - a, &full[slot], pol);
        }
        ++issued;
        prod.advance(p, geo, rp);
      }
    };
#pragma unroll 1
    for (long long r = r0; r < p.s && alive; r += r_step) {
      const long long y = __ldg(p.targets + r);
      if (y == p.ignore_index) continue;
      int ty;
      unsigned toff;
      target_of<EB>(geo, nt, y, ty, toff);
      float m = -INFINITY, se = 0.f, zt = 0.f;
      bool has_t = false;
      RowWalk<EB> cw;
#pragma unroll 1
      for (cw.seek(geo, rp, r, 0); cw.ok; cw.next(geo, rp, r)) {
        top_up();
        if (issued == kc && prod.ok) {  // out of credit for the chunk needed now
          if (!wait_counter_above(&sm.gdone[w], kc - budget)) {
            alive = false;
            break;
          }
          top_up();
        }
        unsigned a, b;
        cw.bounds(a, b);
        const int slot = int(kc % kSSlots);
        if (!mbar_wait_warp(&full[slot], (kc / kSSlots) & 1u)) {
          alive = false;
          break;
        }
        if (lane == 0) st_volatile(&sm.sdone[w], kc + 1);  // these bytes are in L2 now
        stats_chunk_fused<kFVPL>(ring[slot], b - a, lane, m, se, T());
        if (cw.seg == ty && toff >= a && toff < b) {
          has_t = true;
          zt = Elem<T>::load(ring[slot] + (toff - a));
        }
        __syncwarp();
        ++kc;
      }
      if (!alive) break;
      warp_merge_ms(m, se);
      // the mailbox slot of this row last held row n - 2: the grad warps
      // must have taken it (with the credit above this never waits)
      const int buf = int(n & 1u);
      if (n >= 2 && !wait_row_bar(&sm.rowfree[buf], ((n - 2) >> 1) & 1u)) {
        alive = false;
        break;
      }
      // lane 1 posts the row (lane 0 issues this warp's bulk copies).  The
      // other CTAs' copies go by st.async, counted in bytes on their row
      // barriers, so no release at cluster scope (a fence) is on this path:
      // with stores and a release arrival per CTA the pair took 5.59 ms at
      // s = 32768 against 5.16 ms (measured on GB300); s = 16384 (fp32) is
      // unchanged.
      if (lane == 1) {
        // the partial goes to every CTA's mailbox: the grad warps then read
        // all of a row's partials from their own shared memory
        sm.part[buf][crank * kSW + w] = make_float2(m, se);
        if (has_t) sm.tz[buf] = zt;
        if (PAIR) {
#pragma unroll
          for (int c = 0; c < NR; ++c)
            if (unsigned(c) != crank) {
              const uint32_t rb = cluster_addr(&sm.rowdone[buf], unsigned(c));
              st_async_f2(cluster_addr(&sm.part[buf][crank * kSW + w], unsigned(c)), m, se, rb);
              if (has_t) st_async_f32(cluster_addr(&sm.tz[buf], unsigned(c)), zt, rb);
            }
          if (w == 0) {
            // this CTA's barrier also waits for the other CTAs' partials, and
            // for the target logit when another CTA holds it
            const bool t_other = ty >= 0 && !(unsigned(geo.start[ty]) * EB + toff >= cta_lo &&
                                                unsigned(geo.start[ty]) * EB + toff < cta_hi);
            mbar_arrive_expect_tx(&sm.rowdone[buf], unsigned((NR - 1) * kSW * 8 + (t_other ? 4 : 0)));
          } else {
            mbar_arrive_local(&sm.rowdone[buf]);
          }
        } else {
          mbar_arrive_local(&sm.rowdone[buf]);
        }
      }
      ++n;
    }
    if (!alive) {
      if (lane == 0) atomicOr(&p.hdr->error_flag, VPCE_FLAG_WAIT_TIMEOUT);
      for (unsigned i = kc; i < issued; ++i)
        if (!mbar_wait_warp(&full[i % kSSlots], (i / kSSlots) & 1u)) break;
    }
  } else {
    // ---------------- grad warps: logsumexp from the mailbox, pass 2 from L2.
    // A chunk is loaded as soon as the stats partner has received it (so it
    // is in L2), before the row's logsumexp is known; the arithmetic waits
    // for the row's partials.  Loads stay kDSlots - 1 ahead, and a slot is
    // refilled once the store that last used it has read it.
    unsigned char(*ring)[kFChunk] = sm.dring[w];
    uint64_t* full = sm.dfull[w];
    const uint64_t pol = policy_evict_first();
    // the prologue (header, n_valid) may still be running: this kernel is
    // launched as its programmatic dependent, and only the grad warps read
    // what it writes
    grid_dependency_wait();
    const int n_valid = p.hdr->n_valid;
    const float scale_all = p.reduction != VPCE_MEAN ? p.grad : (n_valid > 0 ? p.grad / float(n_valid) : 0.f);
    RowCursor<EB> prod;
    prod.start(p, geo, rp, r0, r_step);
    unsigned kc = 0, issued = 0, n = 0;
    auto issue = [&]() {
      unsigned a, b;
      prod.wk.bounds(a, b);
      const int slot = int(issued % kDSlots);
      if (lane == 0) {
        bulk_wait_read<1>();  // the store of chunk issued - kDSlots has left this slot
        mbar_arrive_expect_tx(&full[slot], b - a);
        bulk_load(ring[slot], prod.wk.addr(a), b - a, &full[slot], pol);
      }
      ++issued;
      prod.advance(p, geo, rp);
    };
    auto top_up = [&]() {
      const unsigned avail = __shfl_sync(kFull, ld_volatile(&sm.sdone[w]), 0);
      while (prod.ok && issued <= kc + kDSlots - 2 && issued < avail) issue();
    };
#pragma unroll 1
    for (long long r = r0; r < p.s && alive; r += r_step) {
      const long long y = __ldg(p.targets + r);
      if (y == p.ignore_index) {
        // ignored row: zeros over this warp's range, nothing read
        for (int i = rp.sa; i < rp.sb; ++i) {
          const unsigned s0 = unsigned(geo.start[i]) * EB;
          const unsigned lo = max(rp.lo, s0), hi = min(rp.hi, unsigned(geo.start[i + 1]) * EB);
          if (hi <= lo) continue;
          uint4* d = reinterpret_cast<uint4*>(const_cast<unsigned char*>(geo.ptr[i]) + r * geo.ld[i] + (lo - s0));
          for (unsigned v = lane; v < (hi - lo) >> 4; v += 32) d[v] = make_uint4(0u, 0u, 0u, 0u);
        }
        if (w == 0 && lane == 0 && crank == 0) {
          p.rowl[r] = 0.f;
          p.lse[r] = 0.f;
          if (p.row_loss) p.row_loss[r] = 0.f;
        }
        continue;
      }
      int ty;
      unsigned toff;
      target_of<EB>(geo, nt, y, ty, toff);
      const bool in_range = ty >= 0;
      const int buf = int(n & 1u);
      top_up();
      if (!wait_row_bar(&sm.rowdone[buf], (n >> 1) & 1u)) {
        alive = false;
        break;
      }
      // every grad warp folds the partials in the same order (CTA rank, then
      // warp; for a pair, one partial per lane and a fixed butterfly): the
      // same lse in every warp of both CTAs
      float M, S, zt;
      if (PAIR) {
        float2 q = make_float2(-INFINITY, 0.f);
        if (lane < NWR) q = sm.part[buf][lane];
        M = q.x;
        S = q.y;
        warp_merge_ms(M, S);
        zt = sm.tz[buf];  // written here by whichever CTA's warp holds the target
      } else {
        M = sm.part[buf][0].x;
        S = sm.part[buf][0].y;
#pragma unroll
        for (int j = 1; j < kSW; ++j) merge_ms(M, S, sm.part[buf][j].x, sm.part[buf][j].y);
        zt = sm.tz[buf];
      }
      __syncwarp();
      // The slot is free once every lane has read it.  The partials' reads
      // returned their values before this point (the fold above used them and
      // the warp has converged), and the target logit's read was issued
      // before it; the slot is written again only after every grad warp of
      // the row's CTAs has arrived and a stats warp has then streamed its part
      // of a whole further row (microseconds, against tens of nanoseconds for
      // a shared-memory load).  So the arrival carries no release: at cluster
      // scope a release made lane 1 wait about 1000 cycles per row for a
      // fence (measured on GB300, s = 32768: 5.73 -> 5.59 ms; s = 16384 fp32:
      // 3.139 -> 3.126 ms).  Lane 0 issues the bulk copies (see the stats side).
      if (lane == 1) {
        if (PAIR) {
#pragma unroll
          for (int c = 0; c < NR; ++c) mbar_arrive_cluster_relaxed(&sm.rowfree[buf], unsigned(c));
        } else {
          mbar_arrive_local(&sm.rowfree[buf]);
        }
      }
      ++n;
      const float lse = in_range ? M + logf(S) : __int_as_float(0x7fc00000);
      if (w == 0 && lane == 0 && crank == 0) {
        const float rl = in_range ? lse - zt : lse;
        p.lse[r] = lse;
        p.rowl[r] = rl;
        if (p.row_loss) p.row_loss[r] = rl;
      }
      const float scale = p.grad_rows != nullptr ? __ldg(p.grad_rows + r) : scale_all;
      const float c = -lse * kLog2e;
      const float cb = folded_offset(c, scale);

      RowWalk<EB> cw;
#pragma unroll 1
      for (cw.seek(geo, rp, r, 0); cw.ok; cw.next(geo, rp, r)) {
        top_up();
        if (issued == kc && prod.ok) issue();  // the stats partner has finished this row: the bytes are in L2
        unsigned a, b;
        cw.bounds(a, b);
        const int slot = int(kc % kDSlots);
        if (!mbar_wait_warp(&full[slot], (kc / kDSlots) & 1u)) {
          alive = false;
          break;
        }
        if (lane == 0) st_volatile(&sm.gdone[w], kc + 1);  // credit back to the stats partner
        unsigned char* sbuf = ring[slot];
        const bool has_t = cw.seg == ty && toff >= a && toff < b;
        float dt = 0.f;
        if (has_t && lane == 0) dt = (ex2(fmaf(Elem<T>::load(sbuf + (toff - a)), kLog2e, c)) - 1.f) * scale;
        __syncwarp();
        grad_chunk_fused<kFVPL>(sbuf, b - a, lane, c, scale, cb, T());
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          if (has_t) {
            Elem<T>::store(sbuf + (toff - a), dt);
            fence_proxy_async_smem();
          }
          bulk_store(cw.addr(a), sbuf, b - a, pol);
          bulk_commit();
        }
        ++kc;
      }
    }
    if (!alive) {
      if (lane == 0) atomicOr(&p.hdr->error_flag, VPCE_FLAG_WAIT_TIMEOUT);
      for (unsigned i = kc; i < issued; ++i)
        if (!mbar_wait_warp(&full[i % kDSlots], (i / kDSlots) & 1u)) break;
    }
    if (lane == 0) bulk_wait_all<0>();  // every dlogits store has landed
  }
  // no CTA leaves while its peer may still reach its mailbox or barriers
  if (PAIR) {
    cluster_sync_all();
    // After a wait that gave up, a partial the other CTA sent (st.async: an
    // asynchronous write, which the barrier above does not order) may still
    // be on its way to this CTA's mailbox, so the CTA stays resident about
    // 100 us longer.  Without an error every byte sent was awaited.
    if (threadIdx.x == 0 && (__ldcg(&p.hdr->error_flag) & VPCE_FLAG_WAIT_TIMEOUT))
      for (int i = 0; i < 100; ++i) __nanosleep(1000);
  }

  // ---- batch loss: the last block sums the per-row losses in a fixed order
  grid_dependency_wait();  // every thread: the header (ticket) is the prologue's
  __threadfence();
  __syncthreads();
  // every copy of this CTA has completed: the stats ring is free scratch
  int* last = reinterpret_cast<int*>(sm.sring[0][0] + 1024);
  if (threadIdx.x == 0) *last = atomicAdd(&p.hdr->ticket, 1u) == gridDim.x - 1;
  __syncthreads();
  if (!*last) return;
  __threadfence();
  // The row losses in a fixed order (see cta_fixed_sum).  The header's count
  // and flag are read at the start, beside those loads: every other CTA set
  // its flag bits before its ticket (fence, then atomic).
  int cnt = 0, flag = 0;
  if (threadIdx.x == 0) {
    cnt = __ldcg(&p.hdr->n_valid);
    flag = __ldcg(&p.hdr->error_flag);
  }
  const double tot = cta_fixed_sum<kFThreads / 32>(p.rowl, p.s, reinterpret_cast<float2*>(sm.sring[0][0]));
  if (threadIdx.x == 0) {
    // a wait that gave up anywhere in the grid leaves rows unfinished: the
    // loss is then NaN rather than a plausible partial sum
    const bool timed_out = (flag & VPCE_FLAG_WAIT_TIMEOUT) != 0;
    p.hdr->loss_sum = tot;
    p.hdr->ticket = 0u;
    if (p.loss_out != nullptr)
      *p.loss_out = timed_out ? __int_as_float(0x7fc00000)
                  : p.reduction != VPCE_MEAN ? float(tot)
                                             : (cnt > 0 ? float(tot / double(cnt)) : __int_as_float(0x7fc00000));
  }
}

}  // namespace

// All shard pointers, row strides and widths 16-byte aligned (the bulk-copy
// engine's requirement for the fused kernels).
bool fused_supported(const ShardSet& sh, int t, int elem) {
  if ((sh.start[t] - sh.start[0]) * elem >= (1LL << 31)) return false;  // row byte offsets are 32-bit
  for (int i = 0; i < t; ++i) {
    const long long wb = (sh.start[i + 1] - sh.start[i]) * elem;
    if ((reinterpret_cast<uintptr_t>(sh.ptr[i]) & 15u) || (sh.ld_bytes[i] & 15) || (wb & 15)) return false;
  }
  return true;
}

cudaError_t set_fused_smem() {
  const int b = int(sizeof(FusedSmem));
  cudaError_t e = cudaSuccess;
  const void* kernels[] = {
      reinterpret_cast<const void*>(stream_fused_kernel<float, 1>),
      reinterpret_cast<const void*>(stream_fused_kernel<float, 2>),
      reinterpret_cast<const void*>(stream_fused_kernel<__nv_bfloat16, 1>),
      reinterpret_cast<const void*>(stream_fused_kernel<__nv_bfloat16, 2>)};
  for (const void* k : kernels)
    if (e == cudaSuccess) e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, b);
  return e;
}

// Pairs of CTAs (one per SM) that fit on the device at once, from the
// occupancy calculator (a GPC with an odd number of free SMs leaves one
// over).  Computed once per device.
int fused_max_clusters(int nr, int sms) {
  static std::mutex mu;
  static int cache[64] = {};
  int dev = 0;
  if (nr == 1) return sms;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
    cudaGetLastError();
    return sms / nr;
  }
  std::lock_guard<std::mutex> lock(mu);
  if (cache[dev] == 0) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(unsigned(nr * (sms / nr)));
    cfg.blockDim = dim3(kFThreads);
    cfg.dynamicSmemBytes = sizeof(FusedSmem);
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeClusterDimension;
    attr.val.clusterDim.x = unsigned(nr);
    attr.val.clusterDim.y = 1;
    attr.val.clusterDim.z = 1;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    int n = 0;
    const cudaError_t e = cudaOccupancyMaxActiveClusters(&n, stream_fused_kernel<__nv_bfloat16, 2>, &cfg);
    if (e != cudaSuccess || n <= 0) {
      cudaGetLastError();
      n = sms / nr;
    }
    cache[dev] = n < sms / nr ? n : sms / nr;
  }
  return cache[dev];
}

// CTAs per row: one up to kPairRowBytes, else a pair.
int fused_cluster(long long row_bytes) { return row_bytes > kPairRowBytes ? 2 : 1; }

// CTAs of the persistent grid: one per SM (a cluster of nr SMs per row, as
// many clusters as fit at once), no more than the rows need.
int fused_grid(long long s, int sms, int nr) {
  const int fit = fused_max_clusters(nr, sms);
  const long long clusters = s < fit ? s : fit;
  return int(nr * clusters);
}

void launch_prep(const long long* targets, long long s, long long V, long long ignore_index, Header* hdr,
                 int reduction, float* loss_out, cudaStream_t st) {
  prep_kernel<<<1, kPrepThreads, 0, st>>>(targets, s, V, ignore_index, hdr, reduction, loss_out);
}

// Chunks of slack per stats warp for rows of row_bytes per CTA: whatever of
// the live budget one row leaves, shared by the kSW stats warps.
unsigned credit_slack(long long row_bytes, bool shared) {
  const long long spare = (long long)(shared ? kLiveBytesPerCtaShared : kLiveBytesPerCta) - row_bytes;
  return spare > 0 ? unsigned(spare / (long long)(kSW * kFChunk)) : 0u;
}

// The streaming fused kernel (expects launch_prep before it): one CTA per SM.
void launch_stream_fused(const ShardSet& sh, bool bf16, int t, long long s, long long V, const long long* targets,
                         long long ignore_index, int reduction, float grad, const float* grad_rows, float* lse,
                         float* rowl, float* row_loss, float* loss_out, Header* hdr, int sms, cudaStream_t st) {
  FusedParams p;
  p.sh = sh;
  p.t = t;
  p.s = s;
  p.V = V;
  p.targets = targets;
  p.ignore_index = ignore_index;
  p.reduction = reduction;
  p.grad = grad;
  p.grad_rows = grad_rows;
  const long long row_bytes = V * (bf16 ? 2 : 4);
  const int nr = fused_cluster(row_bytes);
  p.credit_slack = credit_slack((row_bytes + nr - 1) / nr, nr > 1);
  p.lse = lse;
  p.rowl = rowl;
  p.row_loss = row_loss;
  p.loss_out = loss_out;
  p.hdr = hdr;
  const int grid = fused_grid(s, sms, nr);
  // a programmatic dependent of the prologue: the stats warps start streaming
  // while it counts n_valid
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(unsigned(grid));
  cfg.blockDim = dim3(kFThreads);
  cfg.dynamicSmemBytes = sizeof(FusedSmem);
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = unsigned(nr);
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = nr > 1 ? 2 : 1;
  if (bf16) {
    if (nr == 2) cudaLaunchKernelEx(&cfg, stream_fused_kernel<__nv_bfloat16, 2>, p);
    else cudaLaunchKernelEx(&cfg, stream_fused_kernel<__nv_bfloat16, 1>, p);
  } else {
    if (nr == 2) cudaLaunchKernelEx(&cfg, stream_fused_kernel<float, 2>, p);
    else cudaLaunchKernelEx(&cfg, stream_fused_kernel<float, 1>, p);
  }
}

}  // namespace vpce
