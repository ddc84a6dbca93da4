// In-place backward of the vocab-parallel cross-entropy.
//
// The pages define the forward only; the gradient of the reduced loss is the
// standard one, dlogits_rk = g * (exp(z_rk - lse_r) - [k == y_r]) / n_valid
// for 'mean' (no division for 'sum'; 'none' scales row r by its own g_r),
// zero on ignored rows.  Each (shard, row)
// segment is streamed through shared memory once: the bulk-copy engine loads a
// chunk, the warp turns it into dlogits in place, and the bulk-copy engine
// writes it back over the logits -- one read and one write of the shards.
#include "vpce_chunk.cuh"

namespace vpce {

namespace {

struct ChunkCursorB {
  long long u_end;
  UnitPos pos;
  unsigned off;
  Unit g;
  bool ok;

  // the first unit with chunks at or after the current position
  template <int EB>
  __device__ __forceinline__ void seek(const BackwardParams& p) {
    ok = false;
    for (; pos.u < u_end; pos.step(p.s)) {
      g = make_unit_at(p.sh, pos.shard, pos.row, EB);
      if (g.body == 0) continue;
      if (__ldg(p.targets + g.row) == p.ignore_index) continue;
      off = 0;
      ok = true;
      return;
    }
  }
  template <int EB>
  __device__ __forceinline__ void next(const BackwardParams& p) {
    off += kChunk;
    if (off >= g.body) {
      pos.step(p.s);
      seek<EB>(p);
    }
  }
  __device__ __forceinline__ unsigned bytes() const { return min(unsigned(kChunk), g.body - off); }
  __device__ __forceinline__ const unsigned char* src() const { return g.addr + g.head + off; }
};

template <typename T>
__global__ void __launch_bounds__(kWarps * 32, 1) backward_kernel(const __grid_constant__ BackwardParams p) {
  constexpr int EB = Elem<T>::kBytes;
  extern __shared__ __align__(1024) unsigned char smem[];
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  unsigned char* ring = smem + size_t(warp) * kStages * kChunk;
  uint64_t* bar = reinterpret_cast<uint64_t*>(smem + size_t(kWarps) * kStages * kChunk) + warp * kStages;

  const long long nw = (long long)gridDim.x * kWarps;
  const long long gw = (long long)blockIdx.x * kWarps + warp;
  const long long u0 = p.units * gw / nw;
  const long long u1 = p.units * (gw + 1) / nw;

  if (lane == 0) {
#pragma unroll
    for (int k = 0; k < kStages; ++k) mbar_init(&bar[k], 1);
    fence_mbar_init();
  }
  __syncwarp();
  const uint64_t pol_ld = policy_evict_first();
  const uint64_t pol_st = policy_evict_first();

  // Loads run kStages-1 chunks ahead: the slot of the previous chunk is
  // refilled only once its store has finished reading shared memory.
  ChunkCursorB prod;
  prod.u_end = u1;
  prod.pos.at(u0, p.s);
  prod.seek<EB>(p);
  unsigned issued = 0;
#pragma unroll 1
  for (int k = 0; k < kStages - 1 && prod.ok; ++k) {
    if (lane == 0) {
      mbar_arrive_expect_tx(&bar[k], prod.bytes());
      bulk_load(ring + k * kChunk, prod.src(), prod.bytes(), &bar[k], pol_ld);
    }
    ++issued;
    prod.next<EB>(p);
  }
  // Launched as a programmatic dependent of the kernel ahead (the forward's):
  // everything above reads only the logits and the targets, which the caller
  // leaves as the forward saw them; n_valid and logsumexp are the forward's,
  // read only after it has completed.
  grid_dependency_wait();
  const int n_valid = p.hdr->n_valid;
  const float scale_all =
      p.hdr->reduction != VPCE_MEAN ? p.grad : (n_valid > 0 ? p.grad / float(n_valid) : 0.f);

  unsigned kc = 0;
  bool alive = true;
  UnitPos cur;
  cur.at(u0, p.s);
#pragma unroll 1
  for (; cur.u < u1 && alive; cur.step(p.s)) {
    const Unit g = make_unit_at(p.sh, cur.shard, cur.row, EB);
    const long long y = __ldg(p.targets + g.row);
    const int hn = int(g.head) / EB, tn = int(g.tail) / EB;
    if (y == p.ignore_index) {
      // ignored row: zeros, nothing read
      uint4* body = reinterpret_cast<uint4*>(const_cast<unsigned char*>(g.addr) + g.head);
      const unsigned nv = g.body >> 4;
      for (unsigned k = lane; k < nv; k += 32) body[k] = make_uint4(0u, 0u, 0u, 0u);
      unsigned char* a = const_cast<unsigned char*>(g.addr);
      if (lane < hn) Elem<T>::store(a + lane * EB, 0.f);
      else if (lane >= 16 && lane - 16 < tn) Elem<T>::store(a + g.head + g.body + (lane - 16) * EB, 0.f);
      continue;
    }
    const long long lo = p.sh.start[g.shard], hi = p.sh.start[g.shard + 1];
    const long long tcol = (y >= lo && y < hi) ? (y - lo) : -1;  // target column inside this shard
    const float scale = p.grad_rows != nullptr ? __ldg(p.grad_rows + g.row) : scale_all;
    const float c = -__ldg(p.lse + g.row) * kLog2e;
    const float cb = folded_offset(c, scale);

    // the target element, computed from the original logit before the body
    // is overwritten: (p - 1) * scale
    float dt = 0.f;
    const long long tbyte = tcol >= 0 ? tcol * EB : -1;
    const bool t_in_body = tbyte >= (long long)g.head && tbyte < (long long)(g.head + g.body);
    if (t_in_body && lane == 0) {
      const float zt = Elem<T>::load(g.addr + tbyte);
      dt = (ex2(fmaf(zt, kLog2e, c)) - 1.f) * scale;
    }

    // ragged head / tail elements
    {
      unsigned char* a = const_cast<unsigned char*>(g.addr);
      long long eb = -1;
      if (lane < hn) eb = (long long)lane * EB;
      else if (lane >= 16 && lane - 16 < tn) eb = (long long)(g.head + g.body) + (lane - 16) * EB;
      if (eb >= 0) {
        const float x = Elem<T>::load(a + eb);
        float d = ex2(fmaf(x, kLog2e, c));
        if (eb == tbyte) d -= 1.f;
        Elem<T>::store(a + eb, d * scale);
      }
    }

#pragma unroll 1
    for (unsigned off = 0; off < g.body; off += kChunk) {
      const unsigned n = min(unsigned(kChunk), g.body - off);
      const int slot = int(kc % kStages);
      if (!mbar_wait_warp(&bar[slot], (kc / kStages) & 1u)) {
        alive = false;
        break;
      }
      unsigned char* buf = ring + slot * kChunk;
      grad_chunk<T, kChunk / 512>(buf, n, lane, c, scale, cb);
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
        const long long rel = tbyte - (long long)(g.head + off);
        if (t_in_body && rel >= 0 && rel < (long long)n) {
          Elem<T>::store(buf + rel, dt);
          fence_proxy_async_smem();
        }
        bulk_store(const_cast<unsigned char*>(g.addr) + g.head + off, buf, n, pol_st);
        bulk_commit();
      }
      if (prod.ok) {
        const int ps = int((kc + kStages - 1) % kStages);  // slot of the previous chunk
        if (lane == 0) {
          bulk_wait_read<1>();
          mbar_arrive_expect_tx(&bar[ps], prod.bytes());
          bulk_load(ring + ps * kChunk, prod.src(), prod.bytes(), &bar[ps], pol_ld);
        }
        ++issued;
        prod.next<EB>(p);
      }
      ++kc;
    }
  }

  if (!alive) {
    if (lane == 0) atomicOr(&p.hdr_flags->error_flag, VPCE_FLAG_WAIT_TIMEOUT);
    for (unsigned k = kc; k < issued; ++k) {
      if (!mbar_wait_warp(&bar[k % kStages], (k / kStages) & 1u)) break;
    }
  }
  if (lane == 0) bulk_wait_all<0>();
}

}  // namespace

template <typename T>
void launch_backward(const BackwardParams& p, int grid, cudaStream_t st) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(unsigned(grid));
  cfg.blockDim = dim3(kWarps * 32);
  cfg.dynamicSmemBytes = kRingSmem;
  cfg.stream = st;
  cudaLaunchAttribute attr;
  attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr.val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = &attr;
  cfg.numAttrs = 1;
  cudaLaunchKernelEx(&cfg, backward_kernel<T>, p);
}
template void launch_backward<float>(const BackwardParams&, int, cudaStream_t);
template void launch_backward<__nv_bfloat16>(const BackwardParams&, int, cudaStream_t);

cudaError_t set_backward_smem() {
  cudaError_t e = cudaFuncSetAttribute(backward_kernel<float>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       int(kRingSmem));
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(backward_kernel<__nv_bfloat16>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              int(kRingSmem));
}

}  // namespace vpce
