// Backward of the LM head fused with the loss (vpce_lmhead_backward).
//
// The forward never wrote the logits, so the backward forms them again: per
// chunk of rows, the tensor-core kernel recomputes each logits tile and
// writes dZ = (softmax - onehot) * g as bf16 (the epilogue uses the
// forward's logsumexp and n_valid); then two more tensor-core kernels give
//     dX[chunk]  = sum_i dZ_i W_i          (fp32 accumulators, bf16 out)
//     dW_i      += dZ_i^T X[chunk]         (fp32, accumulated at L2)
// The chunk bounds the dZ scratch to rows x V bf16 (2.1 GB for the default
// 8192 rows at V = 128256; a smaller workspace gives smaller chunks, down to
// 128 rows), the "do not assemble the big tensor" of the CMU notes (§5.5)
// applied to the gradient.
#include "vpce_kernels.cuh"

namespace vpce {

bool launch_gemm_grad(const void* x, long long ld_x, const void* const* w, long long ld_w, int t, long long s,
                      long long h, const long long* vocab_start, const long long* targets, long long ignore_index,
                      const float* lse, const float* grad_rows, float grad, unsigned short* dz, long long ldz,
                      const long long* zcol, Header* hdr, int sms, cudaStream_t st);
bool launch_gemm_stats(const void* x, long long ld_x, const void* const* w, long long ld_w, int t, long long s,
                       long long h, const long long* vocab_start, const long long* targets, long long ignore_index,
                       float2* part, float* tgt, Header* hdr, int sms, int* groups, cudaStream_t st, float* zf,
                       long long ldzf, const long long* zcol);
bool launch_dgrad_x(const unsigned short* dz, long long ldz, const long long* zcol, const void* const* w,
                    long long ld_w, int t, long long R, long long h, const long long* vs, void* dx, long long ld_dx,
                    Header* hdr, int sms, cudaStream_t st);
bool launch_dgrad_w(const unsigned short* dz, long long ldz, const long long* zcol, const void* x, long long ld_x,
                    int t, long long R, long long h, const long long* vs, float* const* dw, long long ld_dw,
                    Header* hdr, int sms, cudaStream_t st);
void launch_prep(const long long* targets, long long s, long long V, long long ignore_index, Header* hdr,
                 int reduction, float* loss_out, cudaStream_t st);

namespace {

constexpr long long kBwdRows = 8192;  // rows per chunk with the suggested workspace
constexpr long long kMinBwdRows = 128;

// The padded row of dZ (and of the kept logits): each shard's columns start
// at a multiple of 8 (16-byte aligned for the TMA), so a row is at most
// round8(V) + 8 * VPCE_MAX_SHARDS columns.
long long padded_ld_bound(long long V) { return (V + 7) / 8 * 8 + 8LL * VPCE_MAX_SHARDS; }

}  // namespace

// Each shard's first column in a padded row; returns the row's width.
long long padded_columns(const long long* vs, int t, long long* zcol) {
  zcol[0] = 0;
  for (int i = 0; i < t; ++i) zcol[i + 1] = zcol[i] + (vs[i + 1] - vs[i] + 7) / 8 * 8;
  return zcol[t];
}

size_t lmhead_bwd_bytes_for(long long rows, long long V, long long /*h*/) {
  return round256(size_t(rows) * size_t(padded_ld_bound(V)) * 2u);
}

size_t lmhead_bwd_workspace_bytes(long long V, long long h) { return lmhead_bwd_bytes_for(kBwdRows, V, h); }
size_t lmhead_bwd_min_workspace_bytes(long long V, long long h) { return lmhead_bwd_bytes_for(kMinBwdRows, V, h); }

// The largest chunk (a multiple of kMinBwdRows, at most kBwdRows) whose
// scratch fits in `bytes`.
long long lmhead_bwd_rows_for(size_t bytes, long long V, long long h) {
  long long r = kBwdRows;
  while (r > kMinBwdRows && lmhead_bwd_bytes_for(r, V, h) > bytes) r -= kMinBwdRows;
  return r;
}

// The two products of one row chunk of R rows, given its bf16 dZ (shard i's
// columns from dz + zcol[i], rows of ldz elements):
//     dX[chunk]  = sum_i dZ_i W_i          (bf16, written)
//     dW_i      += dZ_i^T X[chunk]         (fp32, accumulated)
vpce_status chunk_gemms(const void* xr, long long ld_x, const void* const* w, long long ld_w, int t, long long R,
                        long long h, const long long* vs, const unsigned short* dz, const long long* zcol,
                        long long ldz, void* dxr, long long ld_dx, float* const* dw, long long ld_dw, Header* hdr,
                        int sms, cudaStream_t st) {
  if (!launch_dgrad_x(dz, ldz, zcol, w, ld_w, t, R, h, vs, dxr, ld_dx, hdr, sms, st)) return VPCE_ERR_CUDA;
  if (cudaGetLastError() != cudaSuccess) return VPCE_ERR_CUDA;
  if (!launch_dgrad_w(dz, ldz, zcol, xr, ld_x, t, R, h, vs, dw, ld_dw, hdr, sms, st)) return VPCE_ERR_CUDA;
  return cudaGetLastError() == cudaSuccess ? VPCE_OK : VPCE_ERR_CUDA;
}

// Returns VPCE_OK, VPCE_ERR_CUDA (a launch failed or a tensor map could not
// be encoded).
vpce_status lmhead_backward_run(const void* x, long long ld_x, const void* const* w, long long ld_w, int t,
                                long long s, long long h, const long long* vs, const long long* targets,
                                long long ignore_index, float grad, const float* grad_rows, const float* lse,
                                Header* hdr, void* dx, long long ld_dx, float* const* dw, long long ld_dw, void* ws,
                                size_t ws_bytes, int sms, cudaStream_t st) {
  const long long V = vs[t];
  const long long rows = lmhead_bwd_rows_for(ws_bytes, V, h);
  long long zcol[VPCE_MAX_SHARDS + 1];
  const long long ldz = padded_columns(vs, t, zcol);
  unsigned short* dz = static_cast<unsigned short*>(ws);
  for (long long r0 = 0; r0 < s; r0 += rows) {
    const long long R = s - r0 < rows ? s - r0 : rows;
    const unsigned char* xr = static_cast<const unsigned char*>(x) + r0 * ld_x * 2;
    if (!launch_gemm_grad(xr, ld_x, w, ld_w, t, R, h, vs, targets + r0, ignore_index, lse + r0,
                          grad_rows != nullptr ? grad_rows + r0 : nullptr, grad, dz, ldz, zcol, hdr, sms, st))
      return VPCE_ERR_CUDA;
    if (cudaGetLastError() != cudaSuccess) return VPCE_ERR_CUDA;
    const vpce_status e = chunk_gemms(xr, ld_x, w, ld_w, t, R, h, vs, dz, zcol, ldz,
                                      static_cast<unsigned short*>(dx) + r0 * ld_dx, ld_dx, dw, ld_dw, hdr, sms, st);
    if (e != VPCE_OK) return e;
  }
  return VPCE_OK;
}

// ---------------------------------------------------------------------------
// Forward and backward in one call (vpce_lmhead_forward_backward): per row
// chunk the tensor-core kernel writes the loss statistics and keeps the
// chunk's fp32 logits; one kernel then finishes each row (logsumexp, loss,
// bf16 dZ from the kept logits) and the two tensor-core products follow.  No
// logits are formed twice.
// ---------------------------------------------------------------------------
namespace {

constexpr int kRowThreads = 256;
constexpr int kLossThreads = 1024;

struct TrainRowParams {
  const float2* part;  // [groups][R] (max, sum exp) of the chunk's column groups
  int groups;
  long long R, V;
  int t;
  long long vs[VPCE_MAX_SHARDS + 1];    // shard i holds vocabulary [vs[i], vs[i + 1])
  long long zcol[VPCE_MAX_SHARDS + 1];  // and sits at columns [zcol[i], zcol[i] + w_i) of a padded row
  const float* tgt;    // [R] target logits
  const float* zf;     // [R, ld] fp32 logits, padded per shard
  unsigned short* dz;  // [R, ld] bf16 dlogits, the same layout
  long long ld;        // a multiple of 8
  const long long* targets;
  long long ignore_index;
  const float* grad_rows;  // per-row upstream gradient, or null
  float grad;
  const Header* hdr;       // the batch's n_valid and reduction
  float* lse;
  float* rowl;
  float* row_loss;         // the caller's per-row losses, or null
};

// One row per CTA: the logsumexp of the column groups' partials, folded as
// the combine folds them; the row loss; then dZ = (softmax - onehot) g over
// the row's kept logits, each element as the gradient epilogue forms it.
__global__ void __launch_bounds__(kRowThreads) train_rows_kernel(const __grid_constant__ TrainRowParams p) {
  __shared__ float s_lse;
  const long long rr = blockIdx.x;
  const long long y = p.targets[rr];
  if (threadIdx.x == 0) {
    float rl = 0.f, lse = 0.f;
    if (y == p.ignore_index) {
      rl = 0.f;
    } else if (y < 0 || y >= p.V) {
      rl = lse = __int_as_float(0x7fc00000);
    } else {
      float M = -INFINITY;
      for (int i = 0; i < p.groups; ++i) M = fmaxf(M, p.part[(long long)i * p.R + rr].x);
      float S = 0.f;
      for (int i = 0; i < p.groups; ++i) {
        const float2 q = p.part[(long long)i * p.R + rr];
        S += q.y * expf(q.x - M);
      }
      lse = M + logf(S);
      rl = lse - p.tgt[rr];
    }
    p.lse[rr] = lse;
    p.rowl[rr] = rl;
    if (p.row_loss != nullptr) p.row_loss[rr] = rl;
    s_lse = lse;
  }
  __syncthreads();
  float cb = 0.f, scl = 0.f;  // 0 for ignored rows
  if (y != p.ignore_index) {
    const int nv = p.hdr->n_valid;
    const float sc_all = p.hdr->reduction != VPCE_MEAN ? p.grad : (nv > 0 ? p.grad / float(nv) : 0.f);
    cb = -s_lse * kLog2e;
    scl = p.grad_rows != nullptr ? __ldg(p.grad_rows + rr) : sc_all;
  }
  // the target's column in the padded row (-1: none)
  long long ty = -1;
  if (y >= 0 && y < p.V) {
    int i = 0;
    while (p.vs[i + 1] <= y) ++i;
    ty = p.zcol[i] + (y - p.vs[i]);
  }
  const float* z = p.zf + rr * p.ld;
  unsigned short* d = p.dz + rr * p.ld;
  auto dlogit = [&](float v, long long c) {
    float g = ex2(fmaf(v, kLog2e, cb)) * scl;
    if (c == ty) g -= scl;
    return scl == 0.f ? 0.f : g;
  };
  // the whole padded row: the padding columns were never written and their
  // results are never read
  const long long n4 = p.ld / 4;
  for (long long q = threadIdx.x; q < n4; q += kRowThreads) {
    const float4 v = __ldcs(reinterpret_cast<const float4*>(z) + q);
    const long long c = 4 * q;
    reinterpret_cast<uint2*>(d)[q] =
        make_uint2(pack_bf16x2(dlogit(v.x, c), dlogit(v.y, c + 1)), pack_bf16x2(dlogit(v.z, c + 2), dlogit(v.w, c + 3)));
  }
}

// The batch loss from the per-row losses, summed in a fixed order by one
// CTA (cta_fixed_sum).
__global__ void __launch_bounds__(kLossThreads) train_loss_kernel(const float* rowl, long long s, Header* hdr,
                                                                  float* loss_out) {
  __shared__ float2 sv[kLossThreads / 32];
  const double tot = cta_fixed_sum<kLossThreads / 32>(rowl, s, sv);
  if (threadIdx.x == 0) {
    const int cnt = hdr->n_valid;
    hdr->loss_sum = tot;
    if (loss_out != nullptr)
      *loss_out = hdr->reduction != VPCE_MEAN ? float(tot)
                                              : (cnt > 0 ? float(tot / double(cnt)) : __int_as_float(0x7fc00000));
  }
}

constexpr long long kTrainRows = 8192;  // rows per chunk with the suggested workspace
constexpr long long kMinTrainRows = 128;

struct TrainLayout {
  size_t lse, rowl, part, tgt, zf, dz, total;
  TrainLayout(long long R, long long s, long long V, long long /*h*/) {
    size_t o = 256;  // header
    lse = o;
    o += round256(size_t(s) * 4u);
    rowl = o;
    o += round256(size_t(s) * 4u);
    part = o;
    o += round256(size_t(VPCE_LMHEAD_MAX_GROUPS) * size_t(R) * 8u);
    tgt = o;
    o += round256(size_t(R) * 4u);
    zf = o;
    o += round256(size_t(R) * size_t(padded_ld_bound(V)) * 4u);
    dz = o;
    o += round256(size_t(R) * size_t(padded_ld_bound(V)) * 2u);
    total = o;
  }
};

// the chunk rows a workspace of `bytes` holds (0 when fewer than kMinTrainRows)
long long train_rows_for(size_t bytes, long long s, long long V, long long h) {
  long long r = (s + kMinTrainRows - 1) / kMinTrainRows * kMinTrainRows;
  if (r > kTrainRows) r = kTrainRows;
  if (r < kMinTrainRows) r = kMinTrainRows;
  while (r > kMinTrainRows && TrainLayout(r, s, V, h).total > bytes) r -= kMinTrainRows;
  return TrainLayout(r, s, V, h).total <= bytes ? r : 0;
}

}  // namespace

size_t lmhead_train_workspace_bytes(long long s, long long V, long long h) {
  long long r = (s + kMinTrainRows - 1) / kMinTrainRows * kMinTrainRows;
  if (r > kTrainRows) r = kTrainRows;
  if (r < kMinTrainRows) r = kMinTrainRows;
  return TrainLayout(r, s, V, h).total;
}

size_t lmhead_train_min_workspace_bytes(long long s, long long V, long long h) {
  return TrainLayout(kMinTrainRows, s, V, h).total;
}

// Returns VPCE_OK, VPCE_ERR_WORKSPACE, VPCE_ERR_CUDA (a launch failed or a
// tensor map could not be encoded).
vpce_status lmhead_train_run(const void* x, long long ld_x, const void* const* w, long long ld_w, int t, long long s,
                             long long h, const long long* vs, const long long* targets, long long ignore_index,
                             int reduction, float grad, const float* grad_rows, float* loss_out, float* row_loss_out,
                             void* dx, long long ld_dx, float* const* dw, long long ld_dw, void* ws, size_t ws_bytes,
                             int sms, cudaStream_t st) {
  const long long V = vs[t];
  unsigned char* base = static_cast<unsigned char*>(ws);
  Header* hdr = reinterpret_cast<Header*>(base);
  // the batch's n_valid and reduction in the header, bad targets flagged
  launch_prep(targets, s, V, ignore_index, hdr, reduction, loss_out, st);
  if (cudaGetLastError() != cudaSuccess) return VPCE_ERR_CUDA;
  if (s == 0) return VPCE_OK;
  const long long rows = train_rows_for(ws_bytes, s, V, h);
  if (rows == 0) return VPCE_ERR_WORKSPACE;
  const TrainLayout L(rows, s, V, h);
  float* lse = reinterpret_cast<float*>(base + L.lse);
  float* rowl = reinterpret_cast<float*>(base + L.rowl);
  float* zf = reinterpret_cast<float*>(base + L.zf);
  unsigned short* dz = reinterpret_cast<unsigned short*>(base + L.dz);
  long long zcol[VPCE_MAX_SHARDS + 1];  // each shard's first column in a padded row
  const long long ld = padded_columns(vs, t, zcol);
  for (long long r0 = 0; r0 < s; r0 += rows) {
    const long long R = s - r0 < rows ? s - r0 : rows;
    const unsigned char* xr = static_cast<const unsigned char*>(x) + r0 * ld_x * 2;
    int groups = 1;
    if (!launch_gemm_stats(xr, ld_x, w, ld_w, t, R, h, vs, targets + r0, ignore_index,
                           reinterpret_cast<float2*>(base + L.part), reinterpret_cast<float*>(base + L.tgt), hdr, sms,
                           &groups, st, zf, ld, zcol))
      return VPCE_ERR_CUDA;
    TrainRowParams q;
    q.part = reinterpret_cast<const float2*>(base + L.part);
    q.groups = groups;
    q.R = R;
    q.V = V;
    q.t = t;
    for (int i = 0; i <= t; ++i) {
      q.vs[i] = vs[i];
      q.zcol[i] = zcol[i];
    }
    q.tgt = reinterpret_cast<const float*>(base + L.tgt);
    q.zf = zf;
    q.dz = dz;
    q.ld = ld;
    q.targets = targets + r0;
    q.ignore_index = ignore_index;
    q.grad_rows = grad_rows != nullptr ? grad_rows + r0 : nullptr;
    q.grad = grad;
    q.hdr = hdr;
    q.lse = lse + r0;
    q.rowl = rowl + r0;
    q.row_loss = row_loss_out != nullptr ? row_loss_out + r0 : nullptr;
    train_rows_kernel<<<int(R), kRowThreads, 0, st>>>(q);
    if (cudaGetLastError() != cudaSuccess) return VPCE_ERR_CUDA;
    const vpce_status e = chunk_gemms(xr, ld_x, w, ld_w, t, R, h, vs, dz, zcol, ld,
                                      static_cast<unsigned short*>(dx) + r0 * ld_dx, ld_dx, dw, ld_dw, hdr, sms, st);
    if (e != VPCE_OK) return e;
  }
  train_loss_kernel<<<1, kLossThreads, 0, st>>>(rowl, s, hdr, loss_out);
  return cudaGetLastError() == cudaSuccess ? VPCE_OK : VPCE_ERR_CUDA;
}

}  // namespace vpce
