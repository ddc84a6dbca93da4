// Device twin of the seeded logit generator in vocab_sharded_lm_gb300/synth.py
// (test and benchmark input only; no loss arithmetic).  Each element is drawn
// on its own from a counter: SplitMix64 (Steele, Lea & Flood, OOPSLA 2014)
// outputs 2g and 2g+1 of the value stream, g = row * V + column, feed the
// cosine branch of Box-Muller in float64; the logit is
// float32(sigma * n [+ boost]) and, for bf16 shards, that value rounded to
// nearest-even bfloat16.  Built as its own library, libvpce_synth.so.
#include <cstdint>
#include <cuda_runtime.h>
#include <cuda_bf16.h>

namespace {

constexpr uint64_t kGamma = 0x9E3779B97F4A7C15ull;

__device__ __forceinline__ uint64_t mix64(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

// output n (0-based) of SplitMix64 seeded with key
__device__ __forceinline__ uint64_t splitmix_at(uint64_t key, uint64_t n) { return mix64(key + (n + 1) * kGamma); }

__device__ __forceinline__ double normal_at(uint64_t key, uint64_t g) {
  const uint64_t h1 = splitmix_at(key, 2 * g);
  const uint64_t h2 = splitmix_at(key, 2 * g + 1);
  const double u1 = __dmul_rn(double((h1 >> 11) + 1), 1.0 / 9007199254740992.0);
  const double u2 = __dmul_rn(double(h2 >> 11), 1.0 / 9007199254740992.0);
  const double r = sqrt(__dmul_rn(-2.0, log(u1)));
  return __dmul_rn(r, cos(__dmul_rn(6.283185307179586, u2)));
}

template <typename T>
__device__ __forceinline__ void put(T* p, float v);
template <>
__device__ __forceinline__ void put<float>(float* p, float v) { *p = v; }
template <>
__device__ __forceinline__ void put<__nv_bfloat16>(__nv_bfloat16* p, float v) { *p = __float2bfloat16_rn(v); }

template <typename T>
__global__ void fill_kernel(T* shard, long long s, long long row0, long long col_lo, long long width, long long ld,
                            long long V, uint64_t key, double sigma, const long long* boost_col,
                            double boost_val) {
  const long long n = s * width;
  for (long long e = (long long)blockIdx.x * blockDim.x + threadIdx.x; e < n;
       e += (long long)gridDim.x * blockDim.x) {
    const long long r = e / width;
    const long long j = e - r * width;
    const long long grow = row0 + r;
    const long long gcol = col_lo + j;
    double v = __dmul_rn(normal_at(key, uint64_t(grow) * uint64_t(V) + uint64_t(gcol)), sigma);
    if (boost_col != nullptr && boost_col[grow] == gcol) v = __dadd_rn(v, boost_val);
    put<T>(shard + r * ld + j, __double2float_rn(v));
  }
}

}  // namespace

extern "C" {

// Fill rows [0, s) x columns [0, width) of one shard (row stride ld elements)
// with the logits of global rows row0.. and global columns col_lo.. of a
// vocabulary of V columns.  dtype: 0 = fp32, 1 = bf16.  boost_col: device
// int64 per global row (-1: none) or NULL.  Returns a cudaError_t value.
int vpce_synth_fill(void* shard, int dtype, long long s, long long row0, long long col_lo, long long width,
                    long long ld, long long V, unsigned long long key, double sigma, const long long* boost_col,
                    double boost_val, cudaStream_t stream) {
  if (s <= 0 || width <= 0) return 0;
  const long long n = s * width;
  long long blocks = (n + 255) / 256;
  if (blocks > 152LL * 64) blocks = 152LL * 64;
  if (dtype == 1)
    fill_kernel<__nv_bfloat16><<<int(blocks), 256, 0, stream>>>(static_cast<__nv_bfloat16*>(shard), s, row0,
                                                                col_lo, width, ld, V, key, sigma, boost_col,
                                                                boost_val);
  else
    fill_kernel<float><<<int(blocks), 256, 0, stream>>>(static_cast<float*>(shard), s, row0, col_lo, width, ld,
                                                        V, key, sigma, boost_col, boost_val);
  return int(cudaGetLastError());
}

}  // extern "C"
