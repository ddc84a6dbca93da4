// Per-chunk arithmetic of the streaming kernels: what a warp does with one
// shared-memory chunk of logits.  A chunk is n bytes (a multiple of 16) of
// 16-byte vectors; lane l takes vectors l, l + 32, ...; VPL bounds the vectors
// per lane (chunk capacity / 512 bytes).  The chunk always sits at the start
// of a ring slot of VPL * 512 bytes, and the forms below may read (the fused
// kernel's gradient form also write) the whole slot: only the first n bytes
// ever reach global memory.  Pairs of elements go through packed fp32x2
// instructions; every exponential is one ex2 on the special-function unit.
#pragma once

#include "vpce_kernels.cuh"

namespace vpce {

// 2^(x * log2 e + b) of an element pair, packed
__device__ __forceinline__ f32x2 exp2_pair(f32x2 x, f32x2 l2e, f32x2 b) {
  float e0, e1;
  f2_unpack(f2_fma(x, l2e, b), e0, e1);
  return f2_pack(ex2(e0), ex2(e1));
}

// Running (max m, sum of exp(x - m)) of a lane, updated with VPL of its
// vectors (registers; padding vectors hold -inf): one max over them, one
// rescale, then the sum.
template <int VPL>
__device__ __forceinline__ void stats_vecs(const uint4 (&q)[VPL], float& m, float& sm, __nv_bfloat16) {
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
  const f32x2 l2e = f2_pack(kLog2e, kLog2e);
  const f32x2 nb = f2_pack(-m * kLog2e, -m * kLog2e);
  f32x2 a0 = f2_pack(0.f, 0.f), a1 = a0;
#pragma unroll
  for (int j = 0; j < VPL; ++j) {
    a0 = f2_add(a0, exp2_pair(f2_pack(bf16_lo(q[j].x), bf16_hi(q[j].x)), l2e, nb));
    a1 = f2_add(a1, exp2_pair(f2_pack(bf16_lo(q[j].y), bf16_hi(q[j].y)), l2e, nb));
    a0 = f2_add(a0, exp2_pair(f2_pack(bf16_lo(q[j].z), bf16_hi(q[j].z)), l2e, nb));
    a1 = f2_add(a1, exp2_pair(f2_pack(bf16_lo(q[j].w), bf16_hi(q[j].w)), l2e, nb));
  }
  float s0, s1, s2, s3;
  f2_unpack(a0, s0, s1);
  f2_unpack(a1, s2, s3);
  sm += (s0 + s1) + (s2 + s3);
}

template <int VPL>
__device__ __forceinline__ void stats_vecs(const uint4 (&qu)[VPL], float& m, float& sm, float) {
  const float4(&q)[VPL] = reinterpret_cast<const float4(&)[VPL]>(qu);
  float cm = -INFINITY;
#pragma unroll
  for (int j = 0; j < VPL; ++j) cm = fmaxf(cm, fmaxf(fmaxf(q[j].x, q[j].y), fmaxf(q[j].z, q[j].w)));
  if (cm > m) {
    sm *= ex2((m - cm) * kLog2e);
    m = cm;
  }
  if (m == -INFINITY) return;
  const f32x2 l2e = f2_pack(kLog2e, kLog2e);
  const f32x2 nb = f2_pack(-m * kLog2e, -m * kLog2e);
  f32x2 a0 = f2_pack(0.f, 0.f), a1 = a0;
#pragma unroll
  for (int j = 0; j < VPL; ++j) {
    a0 = f2_add(a0, exp2_pair(f2_pack(q[j].x, q[j].y), l2e, nb));
    a1 = f2_add(a1, exp2_pair(f2_pack(q[j].z, q[j].w), l2e, nb));
  }
  float s0, s1, s2, s3;
  f2_unpack(a0, s0, s1);
  f2_unpack(a1, s2, s3);
  sm += (s0 + s1) + (s2 + s3);
}

// A vector of -inf in the element type (padding for stats_vecs).
__device__ __forceinline__ uint4 neg_inf_vec(__nv_bfloat16) {
  return make_uint4(0xff80ff80u, 0xff80ff80u, 0xff80ff80u, 0xff80ff80u);
}
__device__ __forceinline__ uint4 neg_inf_vec(float) {
  return make_uint4(0xff800000u, 0xff800000u, 0xff800000u, 0xff800000u);
}

// The lane's vectors of a chunk: the whole slot is loaded, and only a short
// chunk (the end of a range) replaces the vectors past n with pad, so a full
// chunk costs no per-vector predicate or select.  Measured on GB300 in the
// fused kernel: s = 32768, V = 256000 (CTA pairs) 5.81 -> 5.72 ms, s = 8192
// 0.662 -> 0.660 ms, s = 4096 0.169 -> 0.167 ms.  The split backward keeps
// its predicated loop (unpredicated, its registers rose from 91 to 249 and
// it ran 1.3% slower).
template <int VPL>
__device__ __forceinline__ void load_slot(const unsigned char* buf, unsigned n, int lane, uint4 (&q)[VPL], uint4 pad) {
  const uint4* v = reinterpret_cast<const uint4*>(buf);
#pragma unroll
  for (int j = 0; j < VPL; ++j) q[j] = v[lane + 32 * j];
  if (n < unsigned(VPL) * 512u) {
    const int nv = int(n >> 4);
#pragma unroll
    for (int j = 0; j < VPL; ++j)
      if (lane + 32 * j >= nv) q[j] = pad;
  }
}

// stats_vecs over the lane's vectors of one shared-memory chunk.
template <int VPL, typename T>
__device__ __forceinline__ void stats_chunk(const unsigned char* buf, unsigned n, int lane, float& m, float& sm, T) {
  uint4 q[VPL];
  load_slot<VPL>(buf, n, lane, q, neg_inf_vec(T()));
  stats_vecs<VPL>(q, m, sm, T());
}

// In place over the lane's vectors: exp(x - lse) * scale.  The exponent
// offset b folds both: b = -lse * log2 e + log2 scale, so one ex2 per element
// and no multiply (used for scale > 0, see grad_chunk).  The
// target element is patched by the caller.
__device__ __forceinline__ uint4 grad_vec(const uint4& w, f32x2 l2e, f32x2 b, __nv_bfloat16) {
  float p0, p1, p2, p3, p4, p5, p6, p7;
  f2_unpack(exp2_pair(f2_pack(bf16_lo(w.x), bf16_hi(w.x)), l2e, b), p0, p1);
  f2_unpack(exp2_pair(f2_pack(bf16_lo(w.y), bf16_hi(w.y)), l2e, b), p2, p3);
  f2_unpack(exp2_pair(f2_pack(bf16_lo(w.z), bf16_hi(w.z)), l2e, b), p4, p5);
  f2_unpack(exp2_pair(f2_pack(bf16_lo(w.w), bf16_hi(w.w)), l2e, b), p6, p7);
  return make_uint4(pack_bf16x2(p0, p1), pack_bf16x2(p2, p3), pack_bf16x2(p4, p5), pack_bf16x2(p6, p7));
}
__device__ __forceinline__ uint4 grad_vec(const uint4& w, f32x2 l2e, f32x2 b, float) {
  float p0, p1, p2, p3;
  f2_unpack(exp2_pair(f2_pack(__uint_as_float(w.x), __uint_as_float(w.y)), l2e, b), p0, p1);
  f2_unpack(exp2_pair(f2_pack(__uint_as_float(w.z), __uint_as_float(w.w)), l2e, b), p2, p3);
  return make_uint4(__float_as_uint(p0), __float_as_uint(p1), __float_as_uint(p2), __float_as_uint(p3));
}

template <typename T, int VPL>
__device__ __forceinline__ void grad_chunk_folded(unsigned char* buf, unsigned n, int lane, float b) {
  uint4* v = reinterpret_cast<uint4*>(buf);
  const int nv = int(n >> 4);
  const f32x2 l2e = f2_pack(kLog2e, kLog2e);
  const f32x2 bb = f2_pack(b, b);
#pragma unroll
  for (int j = 0; j < VPL; ++j) {
    const int idx = lane + 32 * j;
    if (idx < nv) v[idx] = grad_vec(v[idx], l2e, bb, T());
  }
}

// Exponent offset of a row for grad_chunk: -lse * log2 e + log2 scale (only
// used when scale > 0).
__device__ __forceinline__ float folded_offset(float c, float scale) { return scale > 0.f ? c + log2f(scale) : 0.f; }

// exp(x - lse) * scale for every element of the lane's vectors, in place
// (c = -lse * log2 e, cb = folded_offset(c, scale)).  scale > 0 folds into the
// exponent; otherwise (g <= 0, or no valid rows) the product is taken
// explicitly.  The target element is patched by the caller.
template <typename T, int VPL>
__device__ __forceinline__ void grad_chunk(unsigned char* buf, unsigned n, int lane, float c, float scale, float cb) {
  if (scale > 0.f) {
    grad_chunk_folded<T, VPL>(buf, n, lane, cb);
    return;
  }
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

// ---------------------------------------------------------------------------
// Forms for the streaming fused kernel with bf16 logits, whose 16 warps share
// the SM's issue slots with both passes' arithmetic.
//   * One scalar FFMA per element.  The packed form first builds a 64-bit
//     register pair from two unpacked halves, and those moves cost more than
//     the pairing saves.
//   * The gradient loop loads every vector of the lane before it stores any,
//     so the lane's dependent chains overlap (load, exponent, round, store one
//     vector at a time serialises them: the stores may alias the next loads).
// Measured on GB300 at s = 8192, V = 128256: 0.748 -> 0.720 ms per fused
// call.  fp32 logits keep the packed forms and the one-vector loop (their
// float4 vectors already are register pairs; measured 3.65 against 3.74 ms at
// s = 16384, V = 152064), and so do the split kernels (1% faster there).
// ---------------------------------------------------------------------------
template <int VPL>
__device__ __forceinline__ void stats_chunk_fused(const unsigned char* buf, unsigned n, int lane, float& m,
                                                  float& sm, __nv_bfloat16) {
  uint4 q[VPL];
  load_slot<VPL>(buf, n, lane, q, neg_inf_vec(__nv_bfloat16()));
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
  float s0 = 0.f, s1 = 0.f, s2 = 0.f, s3 = 0.f;
#pragma unroll
  for (int j = 0; j < VPL; ++j) {
    s0 += ex2(fmaf(bf16_lo(q[j].x), kLog2e, nb));
    s1 += ex2(fmaf(bf16_hi(q[j].x), kLog2e, nb));
    s2 += ex2(fmaf(bf16_lo(q[j].y), kLog2e, nb));
    s3 += ex2(fmaf(bf16_hi(q[j].y), kLog2e, nb));
    s0 += ex2(fmaf(bf16_lo(q[j].z), kLog2e, nb));
    s1 += ex2(fmaf(bf16_hi(q[j].z), kLog2e, nb));
    s2 += ex2(fmaf(bf16_lo(q[j].w), kLog2e, nb));
    s3 += ex2(fmaf(bf16_hi(q[j].w), kLog2e, nb));
  }
  sm += (s0 + s1) + (s2 + s3);
}

template <int VPL>
__device__ __forceinline__ void stats_chunk_fused(const unsigned char* buf, unsigned n, int lane, float& m,
                                                  float& sm, float) {
  stats_chunk<VPL>(buf, n, lane, m, sm, float());
}

// 2^(x log2 e + b) of every element of a vector, rounded to the element type.
__device__ __forceinline__ uint4 grad_vec_fused(const uint4& w, float b, __nv_bfloat16) {
  const float p0 = ex2(fmaf(bf16_lo(w.x), kLog2e, b)), p1 = ex2(fmaf(bf16_hi(w.x), kLog2e, b));
  const float p2 = ex2(fmaf(bf16_lo(w.y), kLog2e, b)), p3 = ex2(fmaf(bf16_hi(w.y), kLog2e, b));
  const float p4 = ex2(fmaf(bf16_lo(w.z), kLog2e, b)), p5 = ex2(fmaf(bf16_hi(w.z), kLog2e, b));
  const float p6 = ex2(fmaf(bf16_lo(w.w), kLog2e, b)), p7 = ex2(fmaf(bf16_hi(w.w), kLog2e, b));
  return make_uint4(pack_bf16x2(p0, p1), pack_bf16x2(p2, p3), pack_bf16x2(p4, p5), pack_bf16x2(p6, p7));
}
// grad_chunk for the fused kernel: bf16 with a positive scale (the folded
// exponent) loads every vector of the lane, then transforms, then stores;
// everything else is grad_chunk.
template <int VPL>
__device__ __forceinline__ void grad_chunk_fused(unsigned char* buf, unsigned n, int lane, float c, float scale,
                                                 float cb, float) {
  grad_chunk<float, VPL>(buf, n, lane, c, scale, cb);
}

template <int VPL>
__device__ __forceinline__ void grad_chunk_fused(unsigned char* buf, unsigned n, int lane, float c, float scale,
                                                 float cb, __nv_bfloat16) {
  if (!(scale > 0.f)) {
    grad_chunk<__nv_bfloat16, VPL>(buf, n, lane, c, scale, cb);
    return;
  }
  // the whole slot: the bytes past n are never stored to global memory
  uint4* v = reinterpret_cast<uint4*>(buf);
  uint4 q[VPL];
#pragma unroll
  for (int j = 0; j < VPL; ++j) q[j] = v[lane + 32 * j];
#pragma unroll
  for (int j = 0; j < VPL; ++j) q[j] = grad_vec_fused(q[j], cb, __nv_bfloat16());
#pragma unroll
  for (int j = 0; j < VPL; ++j) v[lane + 32 * j] = q[j];
}

}  // namespace vpce
