// Per-chunk arithmetic of the streaming kernels: what a warp does with one
// shared-memory chunk of logits.  A chunk is n bytes (a multiple of 16) of
// 16-byte vectors; lane l takes vectors l, l + 32, ...; VPL bounds the vectors
// per lane (chunk capacity / 512 bytes).
#pragma once

#include "vpce_kernels.cuh"

namespace vpce {

// Running (max m, sum of exp(x - m)) of a lane, updated with the lane's
// vectors of one chunk: one max over the chunk, one rescale, then the sum.
template <int VPL>
__device__ __forceinline__ void stats_chunk(const unsigned char* buf, unsigned n, int lane, float& m, float& sm,
                                            __nv_bfloat16) {
  const uint4* v = reinterpret_cast<const uint4*>(buf);
  const int nv = int(n >> 4);
  uint4 q[VPL];
  const uint4 neg = make_uint4(0xff80ff80u, 0xff80ff80u, 0xff80ff80u, 0xff80ff80u);  // bf16 -inf x8
#pragma unroll
  for (int j = 0; j < VPL; ++j) {
    const int idx = lane + 32 * j;
    q[j] = idx < nv ? v[idx] : neg;
  }
  __nv_bfloat162 mx = __halves2bfloat162(__ushort_as_bfloat16(0xff80), __ushort_as_bfloat16(0xff80));
#pragma unroll
  for (int j = 0; j < VPL; ++j) {
    mx = __hmax2(mx, *reinterpret_cast<const __nv_bfloat162*>(&q[j].x));
    mx = __hmax2(mx, *reinterpret_cast<const __nv_bfloat162*>(&q[j].y));
    mx = __hmax2(mx, *reinterpret_cast<const __nv_bfloat162*>(&q[j].z));
    mx = __hmax2(mx, *reinterpret_cast<const __nv_bfloat162*>(&q[j].w));
  }
  const float cm = fmaxf(__low2float(mx), __high2float(mx));
  if (cm > m) {
    sm *= ex2((m - cm) * kLog2e);
    m = cm;
  }
  if (m == -INFINITY) return;
  const float nb = -m * kLog2e;
  float a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;
#pragma unroll
  for (int j = 0; j < VPL; ++j) {
    float x[8];
    unpack(q[j], x, __nv_bfloat16());
    a0 += ex2(fmaf(x[0], kLog2e, nb));
    a1 += ex2(fmaf(x[1], kLog2e, nb));
    a2 += ex2(fmaf(x[2], kLog2e, nb));
    a3 += ex2(fmaf(x[3], kLog2e, nb));
    a0 += ex2(fmaf(x[4], kLog2e, nb));
    a1 += ex2(fmaf(x[5], kLog2e, nb));
    a2 += ex2(fmaf(x[6], kLog2e, nb));
    a3 += ex2(fmaf(x[7], kLog2e, nb));
  }
  sm += (a0 + a1) + (a2 + a3);
}

template <int VPL>
__device__ __forceinline__ void stats_chunk(const unsigned char* buf, unsigned n, int lane, float& m, float& sm,
                                            float) {
  const float4* v = reinterpret_cast<const float4*>(buf);
  const int nv = int(n >> 4);
  float4 q[VPL];
#pragma unroll
  for (int j = 0; j < VPL; ++j) {
    const int idx = lane + 32 * j;
    q[j] = idx < nv ? v[idx] : make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
  }
  float cm = -INFINITY;
#pragma unroll
  for (int j = 0; j < VPL; ++j) cm = fmaxf(cm, fmaxf(fmaxf(q[j].x, q[j].y), fmaxf(q[j].z, q[j].w)));
  if (cm > m) {
    sm *= ex2((m - cm) * kLog2e);
    m = cm;
  }
  if (m == -INFINITY) return;
  const float nb = -m * kLog2e;
  float a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;
#pragma unroll
  for (int j = 0; j < VPL; ++j) {
    a0 += ex2(fmaf(q[j].x, kLog2e, nb));
    a1 += ex2(fmaf(q[j].y, kLog2e, nb));
    a2 += ex2(fmaf(q[j].z, kLog2e, nb));
    a3 += ex2(fmaf(q[j].w, kLog2e, nb));
  }
  sm += (a0 + a1) + (a2 + a3);
}

// exp(x - lse) * scale for every element of the lane's vectors, in place
// (c = -lse * log2 e).  The target element is patched by the caller.
template <typename T, int VPL>
__device__ __forceinline__ void grad_chunk(unsigned char* buf, unsigned n, int lane, float c, float scale) {
  constexpr int EPV = Elem<T>::kPerVec;
  uint4* v = reinterpret_cast<uint4*>(buf);
  const int nv = int(n >> 4);
#pragma unroll
  for (int j = 0; j < VPL; ++j) {
    const int idx = lane + 32 * j;
    if (idx < nv) {
      float x[EPV];
      unpack(v[idx], x, T());
#pragma unroll
      for (int e = 0; e < EPV; ++e) x[e] = ex2(fmaf(x[e], kLog2e, c)) * scale;
      v[idx] = pack(x, T());
    }
  }
}

}  // namespace vpce
