// C ABI of the vocab-parallel cross-entropy library (declared in include/vpce.h):
// argument validation, launch configuration, and nothing else.  No buffers
// are allocated; every call is stream ordered.
#include <cmath>
#include <cstring>
#include <mutex>

#include "vpce_kernels.cuh"

namespace vpce {
cudaError_t set_backward_smem();
cudaError_t set_fused_smem();
bool fused_supported(const ShardSet& sh, int t, int elem);
void launch_prep(const long long* targets, long long s, long long V, long long ignore_index, Header* hdr,
                 int reduction, float* loss_out, cudaStream_t st);
int fused_cluster(long long row_bytes);
int fused_grid(long long s, int sms, int nr);
void launch_stream_fused(const ShardSet& sh, bool bf16, int t, long long s, long long V, const long long* targets,
                         long long ignore_index, int reduction, float grad, const float* grad_rows, float* lse,
                         float* rowl, float* row_loss, float* loss_out, Header* hdr, int sms, cudaStream_t st);
void launch_fold(const float2* part, int t, long long s, float2* out, cudaStream_t st);
cudaError_t set_gemm_smem();
cudaError_t set_gemm_bwd_smem();
cudaError_t set_embed_smem();
size_t lmhead_bwd_workspace_bytes(long long V, long long h);
size_t lmhead_bwd_min_workspace_bytes(long long V, long long h);
vpce_status lmhead_backward_run(const void* x, long long ld_x, const void* const* w, long long ld_w, int t,
                                long long s, long long h, const long long* vs, const long long* targets,
                                long long ignore_index, float grad, const float* grad_rows, const float* lse,
                                Header* hdr, void* dx, long long ld_dx, float* const* dw, long long ld_dw, void* ws,
                                size_t ws_bytes, int sms, cudaStream_t st);
size_t embed_bwd_workspace_bytes();
void launch_embed_forward(const ShardSet& sh, int t, long long V, long long h, int eb, const long long* ids,
                          long long s, void* out, long long ld_out, int* flag, int sms, cudaStream_t st);
cudaError_t launch_embed_backward(const void* grad, int grad_bf16, long long ld_grad, const long long* ids,
                                  long long s, const ShardSet& gsh, int t, long long V, long long h, void* ws,
                                  int sms, cudaStream_t st);
int gemm_max_shards();
bool launch_gemm_stats(const void* x, long long ld_x, const void* const* w, long long ld_w, int t, long long s,
                       long long h, const long long* vocab_start, const long long* targets, long long ignore_index,
                       float2* part, float* tgt, Header* hdr, int sms, int* groups, cudaStream_t st,
                       float* zf = nullptr, long long ldzf = 0, const long long* zcol = nullptr);
size_t lmhead_train_workspace_bytes(long long s, long long V, long long h);
size_t lmhead_train_min_workspace_bytes(long long s, long long V, long long h);
vpce_status lmhead_train_run(const void* x, long long ld_x, const void* const* w, long long ld_w, int t, long long s,
                             long long h, const long long* vs, const long long* targets, long long ignore_index,
                             int reduction, float grad, const float* grad_rows, float* loss_out, float* row_loss_out,
                             void* dx, long long ld_dx, float* const* dw, long long ld_dw, void* ws, size_t ws_bytes,
                             int sms, cudaStream_t st);

}  // namespace vpce

using namespace vpce;

namespace {

constexpr int kMaxDevices = 64;

struct DeviceInfo {
  int sms = 0;
  bool ready = false;
  vpce_status status = VPCE_OK;
};

DeviceInfo g_dev[kMaxDevices];
std::mutex g_dev_mu;

// Per-device one-time set-up: check the architecture, read the SM count and
// raise the dynamic shared-memory limit of the streaming kernels.
vpce_status device_setup(int* sms) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return VPCE_ERR_CUDA;
  }
  if (dev < 0 || dev >= kMaxDevices) return VPCE_ERR_UNSUPPORTED_DEVICE;
  std::lock_guard<std::mutex> lock(g_dev_mu);
  DeviceInfo& d = g_dev[dev];
  if (!d.ready) {
    int major = 0, minor = 0, sms_ = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms_, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
      cudaGetLastError();
      return VPCE_ERR_CUDA;
    }
    if (major != 10 || minor != 3) {
      d.status = VPCE_ERR_UNSUPPORTED_DEVICE;
    } else if (set_backward_smem() != cudaSuccess ||
               set_fused_smem() != cudaSuccess || set_gemm_smem() != cudaSuccess || set_gemm_bwd_smem() != cudaSuccess ||
               set_embed_smem() != cudaSuccess) {
      cudaGetLastError();
      return VPCE_ERR_CUDA;
    } else {
      d.sms = sms_;
      d.status = VPCE_OK;
    }
    d.ready = true;
  }
  *sms = d.sms;
  return d.status;
}

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// Shared validation of the logits description; fills the geometry.
// from_zero: the shards cover the whole vocabulary (vocab_start[0] = 0);
// otherwise they may be one rank's part of it (vocab_start[0] >= 0).
vpce_status check_logits(const void* const* shards, vpce_dtype dtype, int t, int64_t s,
                         const int64_t* vocab_start, int64_t ld, const int64_t* targets, ShardSet* sh,
                         long long* V, bool from_zero = true) {
  if (dtype != VPCE_FP32 && dtype != VPCE_BF16) return VPCE_ERR_DTYPE;
  if (t < 1 || t > VPCE_MAX_SHARDS || s < 0 || s > (int64_t(1) << 31)) return VPCE_ERR_INVALID_ARG;
  if (shards == nullptr || vocab_start == nullptr) return VPCE_ERR_INVALID_ARG;
  if (s > 0 && targets == nullptr) return VPCE_ERR_INVALID_ARG;
  if (targets != nullptr && !aligned(targets, 8)) return VPCE_ERR_ALIGNMENT;
  const int eb = dtype == VPCE_BF16 ? 2 : 4;
  if (from_zero ? vocab_start[0] != 0 : vocab_start[0] < 0) return VPCE_ERR_INVALID_ARG;
  int64_t wmax = 0;
  for (int i = 0; i < t; ++i) {
    const int64_t w = vocab_start[i + 1] - vocab_start[i];
    if (w < 1) return VPCE_ERR_INVALID_ARG;
    if (w * eb >= (int64_t(1) << 31)) return VPCE_ERR_INVALID_ARG;
    if (w > wmax) wmax = w;
  }
  if (vocab_start[t] >= (int64_t(1) << 31)) return VPCE_ERR_INVALID_ARG;
  if (ld < 0 || (ld > 0 && ld < wmax)) return VPCE_ERR_INVALID_ARG;
  std::memset(sh, 0, sizeof(*sh));
  for (int i = 0; i < t; ++i) {
    if (s > 0 && shards[i] == nullptr) return VPCE_ERR_INVALID_ARG;
    if (!aligned(shards[i], eb)) return VPCE_ERR_ALIGNMENT;
    const int64_t w = vocab_start[i + 1] - vocab_start[i];
    sh->ptr[i] = static_cast<const unsigned char*>(shards[i]);
    sh->ld_bytes[i] = (ld > 0 ? ld : w) * eb;
    sh->start[i] = vocab_start[i];
  }
  sh->start[t] = vocab_start[t];
  *V = vocab_start[t];
  return VPCE_OK;
}

vpce_status check_workspace(const void* ws, size_t bytes, int t, int64_t s) {
  if (ws == nullptr) return VPCE_ERR_INVALID_ARG;
  if (!aligned(ws, 256)) return VPCE_ERR_ALIGNMENT;
  if (bytes < WsLayout(t, s).total) return VPCE_ERR_WORKSPACE;
  return VPCE_OK;
}

int stream_grid(int sms, long long units) {
  const long long want = (units + kWarps - 1) / kWarps;
  return int(want < sms ? (want > 0 ? want : 1) : sms);
}

// Stream-ordered clear of a workspace header's first 16 bytes (n_valid,
// error flag, ticket, reduction).  A memset, not an allocation.
vpce_status clear_header(void* hdr, cudaStream_t cs) {
  if (cudaMemsetAsync(hdr, 0, 16, cs) != cudaSuccess) {
    cudaGetLastError();
    return VPCE_ERR_CUDA;
  }
  return VPCE_OK;
}

vpce_status launch_status() {
  const cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? VPCE_OK : VPCE_ERR_CUDA;
}

// The reduction and the two loss outputs: VPCE_NONE makes the per-row losses
// the result (row_loss_out required unless s = 0, loss_out optional).
vpce_status check_outputs(vpce_reduction reduction, int64_t s, const float* loss_out, const float* row_loss_out) {
  if (reduction != VPCE_MEAN && reduction != VPCE_SUM && reduction != VPCE_NONE) return VPCE_ERR_INVALID_ARG;
  if (reduction == VPCE_NONE ? (row_loss_out == nullptr && s > 0) : loss_out == nullptr)
    return VPCE_ERR_INVALID_ARG;
  if ((loss_out != nullptr && !aligned(loss_out, 4)) || (row_loss_out != nullptr && !aligned(row_loss_out, 4)))
    return VPCE_ERR_ALIGNMENT;
  return VPCE_OK;
}

// Per-row upstream gradients: null means "use the scalar"; otherwise a
// 4-byte aligned device vector with one entry per row.
vpce_status check_grad_rows(const float* grad_rows, int64_t s, bool required) {
  if (grad_rows == nullptr) return (required && s > 0) ? VPCE_ERR_INVALID_ARG : VPCE_OK;
  return aligned(grad_rows, 4) ? VPCE_OK : VPCE_ERR_ALIGNMENT;
}

vpce_status backward_impl(void* const* shards, vpce_dtype dtype, int t, int64_t s, const int64_t* vocab_start,
                          int64_t ld, const int64_t* targets, int64_t ignore_index, float grad_output,
                          const float* grad_rows, const void* workspace, size_t workspace_bytes,
                          vpce_stream_t stream) {
  ShardSet sh;
  long long V = 0;
  vpce_status st = check_logits(reinterpret_cast<const void* const*>(shards), dtype, t, s, vocab_start, ld,
                                targets, &sh, &V, /*from_zero=*/false);
  if (st != VPCE_OK) return st;
  if (!std::isfinite(grad_output)) return VPCE_ERR_INVALID_ARG;
  st = check_workspace(workspace, workspace_bytes, t, s);
  if (st != VPCE_OK) return st;
  int sms = 0;
  st = device_setup(&sms);
  if (st != VPCE_OK) return st;
  if (s == 0) return VPCE_OK;

  const WsLayout L(t, s);
  const unsigned char* ws = static_cast<const unsigned char*>(workspace);
  BackwardParams p;
  p.sh = sh;
  p.s = s;
  p.units = (long long)t * s;
  p.targets = reinterpret_cast<const long long*>(targets);
  p.ignore_index = ignore_index;
  p.lse = reinterpret_cast<const float*>(ws + L.lse);
  p.hdr = reinterpret_cast<const Header*>(ws);
  p.hdr_flags = reinterpret_cast<Header*>(const_cast<unsigned char*>(ws));
  p.grad = grad_output;
  p.grad_rows = grad_rows;
  const int grid = stream_grid(sms, p.units);
  cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  if (dtype == VPCE_BF16) launch_backward<__nv_bfloat16>(p, grid, cs);
  else launch_backward<float>(p, grid, cs);
  return launch_status();
}

vpce_status forward_backward_impl(void* const* shards, vpce_dtype dtype, int t, int64_t s,
                                  const int64_t* vocab_start, int64_t ld, const int64_t* targets,
                                  int64_t ignore_index, vpce_reduction reduction, float grad_output,
                                  const float* grad_rows, float* loss_out, float* row_loss_out, void* workspace,
                                  size_t workspace_bytes, vpce_stream_t stream);

}  // namespace

extern "C" {

size_t vpce_workspace_bytes(int t, int64_t s) {
  if (t < 1 || t > VPCE_MAX_SHARDS || s < 0 || s > (int64_t(1) << 31)) return 0;
  return WsLayout(t, s).total;
}

vpce_status vpce_forward(const void* const* shards, vpce_dtype dtype, int t, int64_t s,
                         const int64_t* vocab_start, int64_t ld, const int64_t* targets, int64_t ignore_index,
                         vpce_reduction reduction, float* loss_out, float* row_loss_out, void* workspace,
                         size_t workspace_bytes, vpce_stream_t stream) {
  ShardSet sh;
  long long V = 0;
  vpce_status st = check_logits(shards, dtype, t, s, vocab_start, ld, targets, &sh, &V);
  if (st != VPCE_OK) return st;
  if ((st = check_outputs(reduction, s, loss_out, row_loss_out)) != VPCE_OK) return st;
  st = check_workspace(workspace, workspace_bytes, t, s);
  if (st != VPCE_OK) return st;
  int sms = 0;
  st = device_setup(&sms);
  if (st != VPCE_OK) return st;

  const WsLayout L(t, s);
  unsigned char* ws = static_cast<unsigned char*>(workspace);
  Header* hdr = reinterpret_cast<Header*>(ws);
  cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  // n_valid, the error flag, the last block's ticket and the per-row arrival
  // counts start at zero, cleared in stream order before any block may set
  // a flag bit (one memset: the counts follow the header)
  if (cudaMemsetAsync(ws, 0, L.part, cs) != cudaSuccess) {
    cudaGetLastError();
    return VPCE_ERR_CUDA;
  }

  if (s > 0) {
    StatsParams p;
    p.sh = sh;
    p.s = s;
    p.units = (long long)t * s;
    p.targets = reinterpret_cast<const long long*>(targets);
    p.ignore_index = ignore_index;
    p.part = reinterpret_cast<float2*>(ws + L.part);
    p.tgt = reinterpret_cast<float*>(ws + L.tgt);
    p.hdr = hdr;
    p.row_cnt = reinterpret_cast<int*>(ws + L.cnt);
    p.t = t;
    p.V = V;
    p.reduction = int(reduction);
    p.lse = reinterpret_cast<float*>(ws + L.lse);
    p.row_loss = row_loss_out;
    p.loss_out = loss_out;
    if (dtype == VPCE_BF16) launch_stats<__nv_bfloat16>(p, sms, cs);
    else launch_stats<float>(p, sms, cs);
    return launch_status();  // the statistics kernel combines the rows and sums the batch
  }
  CombineParams c;
  c.s = s;
  c.t = t;
  c.V = V;
  c.targets = reinterpret_cast<const long long*>(targets);
  c.ignore_index = ignore_index;
  c.reduction = int(reduction);
  c.part = reinterpret_cast<const float2*>(ws + L.part);
  c.tgt = reinterpret_cast<const float*>(ws + L.tgt);
  c.lse = reinterpret_cast<float*>(ws + L.lse);
  c.bsum = reinterpret_cast<double*>(ws + L.bsum);
  c.bcnt = reinterpret_cast<int*>(ws + L.bcnt);
  c.loss_out = loss_out;
  c.row_loss = row_loss_out;
  c.hdr = hdr;
  launch_combine(c, 1, cs);  // s = 0: the empty batch's loss
  return launch_status();
}

vpce_status vpce_backward(void* const* shards, vpce_dtype dtype, int t, int64_t s, const int64_t* vocab_start,
                          int64_t ld, const int64_t* targets, int64_t ignore_index, float grad_output,
                          const void* workspace, size_t workspace_bytes, vpce_stream_t stream) {
  return backward_impl(shards, dtype, t, s, vocab_start, ld, targets, ignore_index, grad_output, nullptr, workspace,
                       workspace_bytes, stream);
}

vpce_status vpce_backward_rows(void* const* shards, vpce_dtype dtype, int t, int64_t s, const int64_t* vocab_start,
                               int64_t ld, const int64_t* targets, int64_t ignore_index, const float* grad_rows,
                               const void* workspace, size_t workspace_bytes, vpce_stream_t stream) {
  const vpce_status st = check_grad_rows(grad_rows, s, true);
  if (st != VPCE_OK) return st;
  return backward_impl(shards, dtype, t, s, vocab_start, ld, targets, ignore_index, 1.f, grad_rows, workspace,
                       workspace_bytes, stream);
}

vpce_status vpce_forward_backward(void* const* shards, vpce_dtype dtype, int t, int64_t s,
                                  const int64_t* vocab_start, int64_t ld, const int64_t* targets,
                                  int64_t ignore_index, vpce_reduction reduction, float grad_output,
                                  float* loss_out, float* row_loss_out, void* workspace, size_t workspace_bytes,
                                  vpce_stream_t stream) {
  return forward_backward_impl(shards, dtype, t, s, vocab_start, ld, targets, ignore_index, reduction, grad_output,
                               nullptr, loss_out, row_loss_out, workspace, workspace_bytes, stream);
}

vpce_status vpce_forward_backward_rows(void* const* shards, vpce_dtype dtype, int t, int64_t s,
                                       const int64_t* vocab_start, int64_t ld, const int64_t* targets,
                                       int64_t ignore_index, vpce_reduction reduction, const float* grad_rows,
                                       float* loss_out, float* row_loss_out, void* workspace,
                                       size_t workspace_bytes, vpce_stream_t stream) {
  const vpce_status st = check_grad_rows(grad_rows, s, true);
  if (st != VPCE_OK) return st;
  return forward_backward_impl(shards, dtype, t, s, vocab_start, ld, targets, ignore_index, reduction, 1.f,
                               grad_rows, loss_out, row_loss_out, workspace, workspace_bytes, stream);
}

}  // extern "C"

namespace {

vpce_status forward_backward_impl(void* const* shards, vpce_dtype dtype, int t, int64_t s,
                                  const int64_t* vocab_start, int64_t ld, const int64_t* targets,
                                  int64_t ignore_index, vpce_reduction reduction, float grad_output,
                                  const float* grad_rows, float* loss_out, float* row_loss_out, void* workspace,
                                  size_t workspace_bytes, vpce_stream_t stream) {
  ShardSet sh;
  long long V = 0;
  vpce_status st = check_logits(reinterpret_cast<const void* const*>(shards), dtype, t, s, vocab_start, ld,
                                targets, &sh, &V);
  if (st != VPCE_OK) return st;
  if ((st = check_outputs(reduction, s, loss_out, row_loss_out)) != VPCE_OK) return st;
  if (!std::isfinite(grad_output)) return VPCE_ERR_INVALID_ARG;
  st = check_workspace(workspace, workspace_bytes, t, s);
  if (st != VPCE_OK) return st;
  int sms = 0;
  st = device_setup(&sms);
  if (st != VPCE_OK) return st;
  const int eb = dtype == VPCE_BF16 ? 2 : 4;
  if (s > 0 && !fused_supported(sh, t, eb)) {
    // rows that are not 16-byte aligned: the two-kernel path (same results)
    st = vpce_forward(reinterpret_cast<const void* const*>(shards), dtype, t, s, vocab_start, ld, targets,
                      ignore_index, reduction, loss_out, row_loss_out, workspace, workspace_bytes, stream);
    if (st != VPCE_OK) return st;
    return backward_impl(shards, dtype, t, s, vocab_start, ld, targets, ignore_index, grad_output, grad_rows,
                         workspace, workspace_bytes, stream);
  }
  const WsLayout L(t, s);
  unsigned char* ws = static_cast<unsigned char*>(workspace);
  const long long* tg = reinterpret_cast<const long long*>(targets);
  Header* hdr = reinterpret_cast<Header*>(ws);
  float* lse = reinterpret_cast<float*>(ws + L.lse);
  float* rowl = reinterpret_cast<float*>(ws + L.tgt);
  cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  launch_prep(tg, s, V, ignore_index, hdr, int(reduction), loss_out, cs);
  if ((st = launch_status()) != VPCE_OK || s == 0) return st;
  launch_stream_fused(sh, dtype == VPCE_BF16, t, s, V, tg, ignore_index, int(reduction), grad_output, grad_rows,
                      lse, rowl, row_loss_out, loss_out, hdr, sms, cs);
  return launch_status();
}

}  // namespace

extern "C" {

vpce_status vpce_fused_plan(vpce_dtype dtype, int t, const int64_t* vocab_start, int64_t s, int* kernel,
                           int* cluster, int* grid) {
  if (kernel == nullptr || cluster == nullptr || grid == nullptr) return VPCE_ERR_INVALID_ARG;
  if (dtype != VPCE_FP32 && dtype != VPCE_BF16) return VPCE_ERR_DTYPE;
  if (t < 1 || t > VPCE_MAX_SHARDS || s < 0 || vocab_start == nullptr || vocab_start[0] != 0)
    return VPCE_ERR_INVALID_ARG;
  for (int i = 0; i < t; ++i)
    if (vocab_start[i + 1] <= vocab_start[i]) return VPCE_ERR_INVALID_ARG;
  int sms = 0;
  const vpce_status st = device_setup(&sms);
  if (st != VPCE_OK) return st;
  const int eb = dtype == VPCE_BF16 ? 2 : 4;
  const int nr = fused_cluster(vocab_start[t] * eb);
  *kernel = 1;
  *cluster = nr;
  *grid = fused_grid(s, sms, nr);
  for (int i = 0; i < t; ++i)
    if (((vocab_start[i + 1] - vocab_start[i]) * eb) & 15) {
      *kernel = 0;
      *grid = 0;
    }
  return VPCE_OK;
}

vpce_status vpce_read_error_flag(const void* workspace, int* flag, vpce_stream_t stream) {
  if (workspace == nullptr || flag == nullptr) return VPCE_ERR_INVALID_ARG;
  if (!aligned(workspace, 256)) return VPCE_ERR_ALIGNMENT;
  cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  const Header* hdr = static_cast<const Header*>(workspace);
  int v = 0;
  if (cudaMemcpyAsync(&v, &hdr->error_flag, sizeof(int), cudaMemcpyDeviceToHost, cs) != cudaSuccess ||
      cudaStreamSynchronize(cs) != cudaSuccess) {
    cudaGetLastError();
    return VPCE_ERR_CUDA;
  }
  *flag = v;
  return VPCE_OK;
}

size_t vpce_lmhead_workspace_bytes(int64_t s) {
  if (s < 0 || s > (int64_t(1) << 31)) return 0;
  return WsLayout(VPCE_LMHEAD_MAX_GROUPS, s).total;
}

vpce_status vpce_lmhead_forward(const void* hidden, int64_t ld_hidden, const void* const* weight_shards,
                                int64_t ld_weight, int t, int64_t s, int64_t h, const int64_t* vocab_start,
                                const int64_t* targets, int64_t ignore_index, vpce_reduction reduction,
                                float* loss_out, float* row_loss_out, void* workspace, size_t workspace_bytes,
                                vpce_stream_t stream) {
  if (t < 1 || t > gemm_max_shards() || s < 0 || s >= (int64_t(1) << 31)) return VPCE_ERR_INVALID_ARG;
  if (h < 64 || h % 64 != 0 || h >= (int64_t(1) << 31)) return VPCE_ERR_INVALID_ARG;
  if (weight_shards == nullptr || vocab_start == nullptr || vocab_start[0] != 0) return VPCE_ERR_INVALID_ARG;
  for (int i = 0; i < t; ++i)
    if (vocab_start[i + 1] <= vocab_start[i]) return VPCE_ERR_INVALID_ARG;
  if (vocab_start[t] >= (int64_t(1) << 31)) return VPCE_ERR_INVALID_ARG;
  const int64_t ldx = ld_hidden == 0 ? h : ld_hidden;
  const int64_t ldw = ld_weight == 0 ? h : ld_weight;
  if (ldx < h || ldw < h) return VPCE_ERR_INVALID_ARG;
  if (s > 0) {
    if (hidden == nullptr || targets == nullptr) return VPCE_ERR_INVALID_ARG;
    for (int i = 0; i < t; ++i)
      if (weight_shards[i] == nullptr) return VPCE_ERR_INVALID_ARG;
  }
  // the tensor-memory-access engine: 16-byte aligned bases and row strides
  if ((hidden != nullptr && !aligned(hidden, 16)) || (ldx * 2) % 16 != 0 || (ldw * 2) % 16 != 0)
    return VPCE_ERR_ALIGNMENT;
  for (int i = 0; i < t; ++i)
    if (weight_shards[i] != nullptr && !aligned(weight_shards[i], 16)) return VPCE_ERR_ALIGNMENT;
  if (targets != nullptr && !aligned(targets, 8)) return VPCE_ERR_ALIGNMENT;
  vpce_status st = check_outputs(reduction, s, loss_out, row_loss_out);
  if (st != VPCE_OK) return st;
  if (workspace == nullptr) return VPCE_ERR_INVALID_ARG;
  if (!aligned(workspace, 256)) return VPCE_ERR_ALIGNMENT;
  if (workspace_bytes < WsLayout(VPCE_LMHEAD_MAX_GROUPS, s).total) return VPCE_ERR_WORKSPACE;
  int sms = 0;
  st = device_setup(&sms);
  if (st != VPCE_OK) return st;

  unsigned char* ws = static_cast<unsigned char*>(workspace);
  Header* hdr = reinterpret_cast<Header*>(ws);
  cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  int groups = 1;
  // partials go where the sharded loss keeps them, [groups][s] (the layout of
  // WsLayout(VPCE_LMHEAD_MAX_GROUPS, s) holds up to that many groups)
  const WsLayout L(VPCE_LMHEAD_MAX_GROUPS, s);
  if ((st = clear_header(hdr, cs)) != VPCE_OK) return st;
  if (s > 0) {
    const int g_sms = sms < VPCE_LMHEAD_MAX_GROUPS ? sms : VPCE_LMHEAD_MAX_GROUPS;
    if (!launch_gemm_stats(hidden, ldx, weight_shards, ldw, t, s, h, reinterpret_cast<const long long*>(vocab_start),
                           reinterpret_cast<const long long*>(targets), ignore_index,
                           reinterpret_cast<float2*>(ws + L.part), reinterpret_cast<float*>(ws + L.tgt), hdr, g_sms,
                           &groups, cs))
      return VPCE_ERR_CUDA;
    if ((st = launch_status()) != VPCE_OK) return st;
  }
  CombineParams c;
  c.s = s;
  c.t = groups;
  c.V = vocab_start[t];
  c.targets = reinterpret_cast<const long long*>(targets);
  c.ignore_index = ignore_index;
  c.reduction = int(reduction);
  c.part = reinterpret_cast<const float2*>(ws + L.part);
  c.tgt = reinterpret_cast<const float*>(ws + L.tgt);
  c.lse = reinterpret_cast<float*>(ws + L.lse);
  c.bsum = reinterpret_cast<double*>(ws + L.bsum);
  c.bcnt = reinterpret_cast<int*>(ws + L.bcnt);
  c.loss_out = loss_out;
  c.row_loss = row_loss_out;
  c.hdr = hdr;
  const long long blocks = s > 0 ? (s + kCombineThreads - 1) / kCombineThreads : 1;
  launch_combine(c, int(blocks), cs);
  return launch_status();
}

vpce_status vpce_partials(const void* const* shards, vpce_dtype dtype, int t, int64_t s, const int64_t* vocab_start,
                          int64_t ld, const int64_t* targets, int64_t ignore_index, float* part_out, float* tgt_out,
                          void* workspace, size_t workspace_bytes, vpce_stream_t stream) {
  ShardSet sh;
  long long V = 0;
  vpce_status st = check_logits(shards, dtype, t, s, vocab_start, ld, targets, &sh, &V, /*from_zero=*/false);
  if (st != VPCE_OK) return st;
  if (s > 0 && (part_out == nullptr || tgt_out == nullptr)) return VPCE_ERR_INVALID_ARG;
  if ((part_out != nullptr && !aligned(part_out, 8)) || (tgt_out != nullptr && !aligned(tgt_out, 4)))
    return VPCE_ERR_ALIGNMENT;
  if ((st = check_workspace(workspace, workspace_bytes, t, s)) != VPCE_OK) return st;
  int sms = 0;
  if ((st = device_setup(&sms)) != VPCE_OK) return st;
  if (s == 0) return VPCE_OK;
  cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  // rows whose target lies in none of these shards contribute 0 to the sum
  if (cudaMemsetAsync(tgt_out, 0, sizeof(float) * size_t(s), cs) != cudaSuccess) {
    cudaGetLastError();
    return VPCE_ERR_CUDA;
  }
  if ((st = clear_header(workspace, cs)) != VPCE_OK) return st;
  StatsParams p;
  p.sh = sh;
  p.s = s;
  p.units = (long long)t * s;
  p.targets = reinterpret_cast<const long long*>(targets);
  p.ignore_index = ignore_index;
  p.part = reinterpret_cast<float2*>(part_out);
  p.tgt = tgt_out;
  p.hdr = reinterpret_cast<Header*>(workspace);
  p.row_cnt = nullptr;  // partials only: the caller exchanges and combines them
  if (dtype == VPCE_BF16) launch_stats<__nv_bfloat16>(p, sms, cs);
  else launch_stats<float>(p, sms, cs);
  return launch_status();
}

vpce_status vpce_fold_partials(const float* part, int t, int64_t s, float* out, vpce_stream_t stream) {
  if (t < 1 || t > VPCE_MAX_SHARDS || s < 0 || s > (int64_t(1) << 31)) return VPCE_ERR_INVALID_ARG;
  if (s > 0 && (part == nullptr || out == nullptr)) return VPCE_ERR_INVALID_ARG;
  if ((part != nullptr && !aligned(part, 8)) || (out != nullptr && !aligned(out, 8))) return VPCE_ERR_ALIGNMENT;
  int sms = 0;
  vpce_status st = device_setup(&sms);
  if (st != VPCE_OK) return st;
  if (s == 0) return VPCE_OK;
  launch_fold(reinterpret_cast<const float2*>(part), t, s, reinterpret_cast<float2*>(out),
              reinterpret_cast<cudaStream_t>(stream));
  return launch_status();
}

vpce_status vpce_combine_partials(const float* part, int n_part, const float* tgt, int64_t s, int64_t V,
                                  const int64_t* targets, int64_t ignore_index, vpce_reduction reduction,
                                  float* loss_out, float* row_loss_out, int t_local, void* workspace,
                                  size_t workspace_bytes, vpce_stream_t stream) {
  if (n_part < 1 || s < 0 || s > (int64_t(1) << 31) || V < 1 || V >= (int64_t(1) << 31)) return VPCE_ERR_INVALID_ARG;
  if (t_local < 1 || t_local > VPCE_MAX_SHARDS) return VPCE_ERR_INVALID_ARG;
  if (s > 0 && (part == nullptr || tgt == nullptr || targets == nullptr)) return VPCE_ERR_INVALID_ARG;
  if ((part != nullptr && !aligned(part, 8)) || (tgt != nullptr && !aligned(tgt, 4)) ||
      (targets != nullptr && !aligned(targets, 8)))
    return VPCE_ERR_ALIGNMENT;
  vpce_status st = check_outputs(reduction, s, loss_out, row_loss_out);
  if (st != VPCE_OK) return st;
  if ((st = check_workspace(workspace, workspace_bytes, t_local, s)) != VPCE_OK) return st;
  int sms = 0;
  if ((st = device_setup(&sms)) != VPCE_OK) return st;
  cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  // a fresh header: n_valid, error flag and ticket start at zero
  if ((st = clear_header(workspace, cs)) != VPCE_OK) return st;
  const WsLayout L(t_local, s);
  unsigned char* ws = static_cast<unsigned char*>(workspace);
  CombineParams c;
  c.s = s;
  c.t = n_part;
  c.V = V;
  c.targets = reinterpret_cast<const long long*>(targets);
  c.ignore_index = ignore_index;
  c.reduction = int(reduction);
  c.part = reinterpret_cast<const float2*>(part);
  c.tgt = tgt;
  c.lse = reinterpret_cast<float*>(ws + L.lse);
  c.bsum = reinterpret_cast<double*>(ws + L.bsum);
  c.bcnt = reinterpret_cast<int*>(ws + L.bcnt);
  c.loss_out = loss_out;
  c.row_loss = row_loss_out;
  c.hdr = reinterpret_cast<Header*>(ws);
  const long long blocks = s > 0 ? (s + kCombineThreads - 1) / kCombineThreads : 1;
  launch_combine(c, int(blocks), cs);
  return launch_status();
}

size_t vpce_lmhead_backward_workspace_bytes(int64_t V, int64_t h) {
  if (V < 1 || h < 1) return 0;
  return lmhead_bwd_workspace_bytes(V, h);
}

vpce_status vpce_lmhead_backward(const void* hidden, int64_t ld_hidden, const void* const* weight_shards,
                                 int64_t ld_weight, int t, int64_t s, int64_t h, const int64_t* vocab_start,
                                 const int64_t* targets, int64_t ignore_index, float grad_output,
                                 const float* grad_rows, const void* fwd_workspace, size_t fwd_workspace_bytes,
                                 void* grad_hidden, int64_t ld_grad_hidden, float* const* grad_weight_shards,
                                 int64_t ld_grad_weight, void* workspace, size_t workspace_bytes,
                                 vpce_stream_t stream) {
  if (t < 1 || t > gemm_max_shards() || s < 0 || s >= (int64_t(1) << 31)) return VPCE_ERR_INVALID_ARG;
  if (h < 64 || h % 64 != 0 || h >= (int64_t(1) << 31)) return VPCE_ERR_INVALID_ARG;
  if (weight_shards == nullptr || grad_weight_shards == nullptr || vocab_start == nullptr || vocab_start[0] != 0)
    return VPCE_ERR_INVALID_ARG;
  for (int i = 0; i < t; ++i)
    if (vocab_start[i + 1] <= vocab_start[i]) return VPCE_ERR_INVALID_ARG;
  if (vocab_start[t] >= (int64_t(1) << 31)) return VPCE_ERR_INVALID_ARG;
  if (!std::isfinite(grad_output)) return VPCE_ERR_INVALID_ARG;
  const int64_t ldx = ld_hidden == 0 ? h : ld_hidden;
  const int64_t ldw = ld_weight == 0 ? h : ld_weight;
  const int64_t ldgx = ld_grad_hidden == 0 ? h : ld_grad_hidden;
  const int64_t ldgw = ld_grad_weight == 0 ? h : ld_grad_weight;
  if (ldx < h || ldw < h || ldgx < h || ldgw < h) return VPCE_ERR_INVALID_ARG;
  if (s > 0) {
    if (hidden == nullptr || targets == nullptr || grad_hidden == nullptr) return VPCE_ERR_INVALID_ARG;
    for (int i = 0; i < t; ++i)
      if (weight_shards[i] == nullptr || grad_weight_shards[i] == nullptr) return VPCE_ERR_INVALID_ARG;
  }
  // the tensor-memory-access engine reads X, W_i and adds into dW_i: 16-byte
  // aligned bases and row strides
  if ((hidden != nullptr && !aligned(hidden, 16)) || (ldx * 2) % 16 != 0 || (ldw * 2) % 16 != 0 ||
      (ldgw * 4) % 16 != 0)
    return VPCE_ERR_ALIGNMENT;
  for (int i = 0; i < t; ++i) {
    if (weight_shards[i] != nullptr && !aligned(weight_shards[i], 16)) return VPCE_ERR_ALIGNMENT;
    if (grad_weight_shards[i] != nullptr && !aligned(grad_weight_shards[i], 16)) return VPCE_ERR_ALIGNMENT;
  }
  if ((grad_hidden != nullptr && !aligned(grad_hidden, 2)) || (targets != nullptr && !aligned(targets, 8)) ||
      (grad_rows != nullptr && !aligned(grad_rows, 4)))
    return VPCE_ERR_ALIGNMENT;
  if (fwd_workspace == nullptr || workspace == nullptr) return VPCE_ERR_INVALID_ARG;
  if (!aligned(fwd_workspace, 256) || !aligned(workspace, 256)) return VPCE_ERR_ALIGNMENT;
  if (fwd_workspace_bytes < WsLayout(VPCE_LMHEAD_MAX_GROUPS, s).total ||
      workspace_bytes < lmhead_bwd_min_workspace_bytes(vocab_start[t], h))
    return VPCE_ERR_WORKSPACE;
  int sms = 0;
  vpce_status st = device_setup(&sms);
  if (st != VPCE_OK) return st;
  if (s == 0) return VPCE_OK;
  const WsLayout L(VPCE_LMHEAD_MAX_GROUPS, s);
  const unsigned char* fws = static_cast<const unsigned char*>(fwd_workspace);
  const int g_sms = sms < VPCE_LMHEAD_MAX_GROUPS ? sms : VPCE_LMHEAD_MAX_GROUPS;
  return lmhead_backward_run(hidden, ldx, weight_shards, ldw, t, s, h, reinterpret_cast<const long long*>(vocab_start),
                             reinterpret_cast<const long long*>(targets), ignore_index, grad_output, grad_rows,
                             reinterpret_cast<const float*>(fws + L.lse),
                             reinterpret_cast<Header*>(const_cast<unsigned char*>(fws)), grad_hidden, ldgx,
                             grad_weight_shards, ldgw, workspace, workspace_bytes, g_sms,
                             reinterpret_cast<cudaStream_t>(stream));
}

size_t vpce_lmhead_forward_backward_workspace_bytes(int64_t s, int64_t V, int64_t h) {
  if (s < 0 || s >= (int64_t(1) << 31) || V < 1 || h < 1) return 0;
  return lmhead_train_workspace_bytes(s, V, h);
}

vpce_status vpce_lmhead_forward_backward(const void* hidden, int64_t ld_hidden, const void* const* weight_shards,
                                         int64_t ld_weight, int t, int64_t s, int64_t h, const int64_t* vocab_start,
                                         const int64_t* targets, int64_t ignore_index, vpce_reduction reduction,
                                         float grad_output, const float* grad_rows, float* loss_out,
                                         float* row_loss_out, void* grad_hidden, int64_t ld_grad_hidden,
                                         float* const* grad_weight_shards, int64_t ld_grad_weight, void* workspace,
                                         size_t workspace_bytes, vpce_stream_t stream) {
  if (t < 1 || t > gemm_max_shards() || s < 0 || s >= (int64_t(1) << 31)) return VPCE_ERR_INVALID_ARG;
  if (h < 64 || h % 64 != 0 || h >= (int64_t(1) << 31)) return VPCE_ERR_INVALID_ARG;
  if (weight_shards == nullptr || grad_weight_shards == nullptr || vocab_start == nullptr || vocab_start[0] != 0)
    return VPCE_ERR_INVALID_ARG;
  for (int i = 0; i < t; ++i)
    if (vocab_start[i + 1] <= vocab_start[i]) return VPCE_ERR_INVALID_ARG;
  if (vocab_start[t] >= (int64_t(1) << 31)) return VPCE_ERR_INVALID_ARG;
  if (!std::isfinite(grad_output)) return VPCE_ERR_INVALID_ARG;
  if (reduction == VPCE_NONE && s > 0 && grad_rows == nullptr) return VPCE_ERR_INVALID_ARG;
  const int64_t ldx = ld_hidden == 0 ? h : ld_hidden;
  const int64_t ldw = ld_weight == 0 ? h : ld_weight;
  const int64_t ldgx = ld_grad_hidden == 0 ? h : ld_grad_hidden;
  const int64_t ldgw = ld_grad_weight == 0 ? h : ld_grad_weight;
  if (ldx < h || ldw < h || ldgx < h || ldgw < h) return VPCE_ERR_INVALID_ARG;
  if (s > 0) {
    if (hidden == nullptr || targets == nullptr || grad_hidden == nullptr) return VPCE_ERR_INVALID_ARG;
    for (int i = 0; i < t; ++i)
      if (weight_shards[i] == nullptr || grad_weight_shards[i] == nullptr) return VPCE_ERR_INVALID_ARG;
  }
  // the tensor-memory-access engine reads X, W_i and adds into dW_i: 16-byte
  // aligned bases and row strides
  if ((hidden != nullptr && !aligned(hidden, 16)) || (ldx * 2) % 16 != 0 || (ldw * 2) % 16 != 0 ||
      (ldgw * 4) % 16 != 0)
    return VPCE_ERR_ALIGNMENT;
  for (int i = 0; i < t; ++i) {
    if (weight_shards[i] != nullptr && !aligned(weight_shards[i], 16)) return VPCE_ERR_ALIGNMENT;
    if (grad_weight_shards[i] != nullptr && !aligned(grad_weight_shards[i], 16)) return VPCE_ERR_ALIGNMENT;
  }
  if ((grad_hidden != nullptr && !aligned(grad_hidden, 2)) || (targets != nullptr && !aligned(targets, 8)) ||
      (grad_rows != nullptr && !aligned(grad_rows, 4)))
    return VPCE_ERR_ALIGNMENT;
  vpce_status st = check_outputs(reduction, s, loss_out, row_loss_out);
  if (st != VPCE_OK) return st;
  if (workspace == nullptr) return VPCE_ERR_INVALID_ARG;
  if (!aligned(workspace, 256)) return VPCE_ERR_ALIGNMENT;
  if (workspace_bytes < lmhead_train_min_workspace_bytes(s, vocab_start[t], h)) return VPCE_ERR_WORKSPACE;
  int sms = 0;
  if ((st = device_setup(&sms)) != VPCE_OK) return st;
  const int g_sms = sms < VPCE_LMHEAD_MAX_GROUPS ? sms : VPCE_LMHEAD_MAX_GROUPS;
  return lmhead_train_run(hidden, ldx, weight_shards, ldw, t, s, h, reinterpret_cast<const long long*>(vocab_start),
                          reinterpret_cast<const long long*>(targets), ignore_index, int(reduction), grad_output,
                          grad_rows, loss_out, row_loss_out, grad_hidden, ldgx, grad_weight_shards, ldgw, workspace,
                          workspace_bytes, g_sms, reinterpret_cast<cudaStream_t>(stream));
}

// Shard geometry of a [w_i, h] table split by vocabulary (row stride ld
// elements of eb bytes); checks the offsets and the pointers.
static vpce_status split_table(const void* const* shards, int t, const int64_t* vocab_start, int64_t ld, int eb,
                                bool need_ptrs, ShardSet* sh) {
  if (shards == nullptr || vocab_start == nullptr || vocab_start[0] != 0) return VPCE_ERR_INVALID_ARG;
  std::memset(sh, 0, sizeof(*sh));
  for (int i = 0; i < t; ++i) {
    if (vocab_start[i + 1] <= vocab_start[i]) return VPCE_ERR_INVALID_ARG;
    if (need_ptrs && shards[i] == nullptr) return VPCE_ERR_INVALID_ARG;
    if (!aligned(shards[i], size_t(eb))) return VPCE_ERR_ALIGNMENT;
    sh->ptr[i] = static_cast<const unsigned char*>(shards[i]);
    sh->ld_bytes[i] = ld * eb;
    sh->start[i] = vocab_start[i];
  }
  sh->start[t] = vocab_start[t];
  return VPCE_OK;
}

vpce_status vpce_embedding_forward(const void* const* table_shards, vpce_dtype dtype, int t,
                                   const int64_t* vocab_start, int64_t h, int64_t ld_table, const int64_t* ids,
                                   int64_t s, void* out, int64_t ld_out, int* flag_out, vpce_stream_t stream) {
  if (dtype != VPCE_FP32 && dtype != VPCE_BF16) return VPCE_ERR_DTYPE;
  if (t < 1 || t > VPCE_MAX_SHARDS || s < 0 || h < 1) return VPCE_ERR_INVALID_ARG;
  const int eb = dtype == VPCE_BF16 ? 2 : 4;
  const int64_t ldt = ld_table == 0 ? h : ld_table;
  const int64_t ldo = ld_out == 0 ? h : ld_out;
  if (ldt < h || ldo < h) return VPCE_ERR_INVALID_ARG;
  ShardSet sh;
  vpce_status st = split_table(table_shards, t, vocab_start, ldt, eb, s > 0, &sh);
  if (st != VPCE_OK) return st;
  if (s > 0 && (ids == nullptr || out == nullptr)) return VPCE_ERR_INVALID_ARG;
  if ((ids != nullptr && !aligned(ids, 8)) || (out != nullptr && !aligned(out, size_t(eb))) ||
      (flag_out != nullptr && !aligned(flag_out, 4)))
    return VPCE_ERR_ALIGNMENT;
  int sms = 0;
  st = device_setup(&sms);
  if (st != VPCE_OK) return st;
  cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  if (flag_out != nullptr && cudaMemsetAsync(flag_out, 0, sizeof(int), cs) != cudaSuccess) {
    cudaGetLastError();
    return VPCE_ERR_CUDA;
  }
  if (s == 0) return VPCE_OK;
  launch_embed_forward(sh, t, vocab_start[t], h, eb, reinterpret_cast<const long long*>(ids), s, out, ldo,
                       flag_out, sms, cs);
  return launch_status();
}

size_t vpce_embedding_backward_workspace_bytes(void) { return embed_bwd_workspace_bytes(); }

vpce_status vpce_embedding_backward(const void* grad_out, vpce_dtype grad_dtype, int64_t ld_grad,
                                    const int64_t* ids, int64_t s, float* const* grad_shards, int t,
                                    const int64_t* vocab_start, int64_t h, int64_t ld_grad_table, void* workspace,
                                    size_t workspace_bytes, vpce_stream_t stream) {
  if (grad_dtype != VPCE_FP32 && grad_dtype != VPCE_BF16) return VPCE_ERR_DTYPE;
  if (t < 1 || t > VPCE_MAX_SHARDS || s < 0 || h < 4 || h % 4 != 0) return VPCE_ERR_INVALID_ARG;
  const int eb = grad_dtype == VPCE_BF16 ? 2 : 4;
  const int64_t ldg = ld_grad == 0 ? h : ld_grad;
  const int64_t ldt = ld_grad_table == 0 ? h : ld_grad_table;
  if (ldg < h || ldt < h) return VPCE_ERR_INVALID_ARG;
  ShardSet gsh;
  vpce_status st = split_table(reinterpret_cast<const void* const*>(grad_shards), t, vocab_start, ldt, 4, s > 0,
                                &gsh);
  if (st != VPCE_OK) return st;
  for (int i = 0; i < t; ++i)
    if (grad_shards[i] != nullptr && !aligned(grad_shards[i], 16)) return VPCE_ERR_ALIGNMENT;
  if ((ldt * 4) % 16 != 0) return VPCE_ERR_ALIGNMENT;
  if (s > 0 && (grad_out == nullptr || ids == nullptr)) return VPCE_ERR_INVALID_ARG;
  if ((grad_out != nullptr && !aligned(grad_out, 16)) || (ldg * eb) % 16 != 0) return VPCE_ERR_ALIGNMENT;
  if (ids != nullptr && !aligned(ids, 8)) return VPCE_ERR_ALIGNMENT;
  if (workspace == nullptr) return VPCE_ERR_INVALID_ARG;
  if (!aligned(workspace, 256)) return VPCE_ERR_ALIGNMENT;
  if (workspace_bytes < embed_bwd_workspace_bytes()) return VPCE_ERR_WORKSPACE;
  int sms = 0;
  st = device_setup(&sms);
  if (st != VPCE_OK) return st;
  if (s == 0) return VPCE_OK;
  const cudaError_t e = launch_embed_backward(grad_out, grad_dtype == VPCE_BF16, ldg,
                                              reinterpret_cast<const long long*>(ids), s, gsh, t, vocab_start[t],
                                              h, workspace, sms, reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? VPCE_OK : VPCE_ERR_CUDA;
}

const char* vpce_status_string(vpce_status status) {
  switch (status) {
    case VPCE_OK: return "VPCE_OK";
    case VPCE_ERR_INVALID_ARG: return "VPCE_ERR_INVALID_ARG: invalid argument";
    case VPCE_ERR_ALIGNMENT: return "VPCE_ERR_ALIGNMENT: misaligned pointer";
    case VPCE_ERR_DTYPE: return "VPCE_ERR_DTYPE: unsupported dtype";
    case VPCE_ERR_WORKSPACE: return "VPCE_ERR_WORKSPACE: workspace too small";
    case VPCE_ERR_CUDA: return "VPCE_ERR_CUDA: CUDA runtime or launch error";
    case VPCE_ERR_UNSUPPORTED_DEVICE: return "VPCE_ERR_UNSUPPORTED_DEVICE: needs a compute capability 10.3 GPU";
  }
  return "VPCE_ERR_UNKNOWN";
}

}  // extern "C"
