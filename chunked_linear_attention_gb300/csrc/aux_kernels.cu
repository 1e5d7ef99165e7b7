// Bandwidth-bound kernels around the GEMMs: fast-weight initialisation and
// operand copies, the update + row L2-normalisation (eq 5/6 of the LaCT
// notes: W <- L2-Normalize(W - U) along the input dimension), the eta
// scaling of linear-attention values, and the prefix of per-chunk
// linear-attention states.
#include "common.cuh"
#include "launch.h"
#include "linattn_kernels.h"

namespace ttt {

// ------------------------------------------------------------ init weights
__global__ void init_weights_kernel(const float* __restrict__ init, int init_per_batch,
                                    float* __restrict__ master, __nv_bfloat16* __restrict__ work,
                                    int H, long long per_mat, long long total) {
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < total;
       i += (long long)gridDim.x * blockDim.x) {
    const long long bh = i / per_mat, e = i - bh * per_mat;
    const long long src = (init_per_batch ? bh : bh % H) * per_mat + e;
    const float w = init[src];
    master[i] = w;
    if (work) work[i] = __float2bfloat16_rn(w);
  }
}

cudaError_t launch_init_weights(const MatSet& m, int B, int H, cudaStream_t stream) {
  const long long per = (long long)m.rows * m.cols;
  const long long total = per * B * H;
  const int threads = 256;
  long long blocks = (total + threads - 1) / threads;
  if (blocks > 152 * 16) blocks = 152 * 16;
  init_weights_kernel<<<(int)blocks, threads, 0, stream>>>(
      m.init, m.init_per_batch, m.master, static_cast<__nv_bfloat16*>(m.work), H, per, total);
  return cudaGetLastError();
}

// ------------------------------------------------------------ update + normalise
// One warp per matrix row.  Rows hold at most 1024 entries (32 per lane).
struct NormArgs {
  MatSet sets[3];
  int nsets;
  int BH;
  int l2norm;
  long long rows_before[4];  // prefix of BH*rows over the sets
};

__global__ void __launch_bounds__(256) update_normalize_kernel(const __grid_constant__ NormArgs a) {
  const long long gw = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (gw >= a.rows_before[a.nsets]) return;
  int s = 0;
  while (s + 1 < a.nsets && gw >= a.rows_before[s + 1]) ++s;
  const MatSet& m = a.sets[s];
  const long long row = gw - a.rows_before[s];
  const long long off = row * m.cols;
  float* w = m.master + off;
  const float* u = m.update + off;
  float vals[32];
  float ss = 0.f;
#pragma unroll
  for (int i = 0; i < 32; ++i) {
    const int c = lane + 32 * i;
    float x = 0.f;
    if (c < m.cols) x = w[c] - u[c];
    vals[i] = x;
    ss += x * x;
  }
  float scale = 1.f;
  if (a.l2norm) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
    scale = 1.0f / fmaxf(sqrtf(ss), 1e-12f);
  }
  __nv_bfloat16* wb = m.work ? static_cast<__nv_bfloat16*>(m.work) + off : nullptr;
#pragma unroll
  for (int i = 0; i < 32; ++i) {
    const int c = lane + 32 * i;
    if (c < m.cols) {
      const float y = vals[i] * scale;
      w[c] = y;
      if (wb) wb[c] = __float2bfloat16_rn(y);
    }
  }
}

cudaError_t launch_update_normalize(const MatSet* sets, int nsets, int BH, int l2norm,
                                    cudaStream_t stream) {
  NormArgs a{};
  a.nsets = nsets;
  a.BH = BH;
  a.l2norm = l2norm;
  a.rows_before[0] = 0;
  for (int i = 0; i < nsets; ++i) {
    a.sets[i] = sets[i];
    a.rows_before[i + 1] = a.rows_before[i] + (long long)BH * sets[i].rows;
  }
  const long long warps = a.rows_before[nsets];
  const long long blocks = (warps * 32 + 255) / 256;
  update_normalize_kernel<<<(int)(blocks > 0 ? blocks : 1), 256, 0, stream>>>(a);
  return cudaGetLastError();
}

// ------------------------------------------------------------ gradient norms
// out[s * BH + h] = fixed-order sum of the nslot partials of matrix (s, h),
// for s = 0..2 and h in [h0, h0 + nh): one warp per matrix.
__global__ void normsq_reduce_kernel(const float* __restrict__ part, int nslot,
                                     float* __restrict__ out, int BH, int h0, int nh) {
  const int w = (int)((blockIdx.x * blockDim.x + threadIdx.x) >> 5);
  if (w >= 3 * nh) return;
  const int z = (w / nh) * BH + h0 + w % nh;
  const float s = sum_partials_warp(part + (long long)z * nslot, nslot);
  if ((threadIdx.x & 31) == 0) out[z] = s;
}

cudaError_t launch_normsq_reduce(const float* part, int nslot, float* out, int BH, int h0,
                                 int nh, cudaStream_t stream) {
  if (nh <= 0) return cudaSuccess;
  const int blocks = (3 * nh * 32 + 255) / 256;
  normsq_reduce_kernel<<<blocks, 256, 0, stream>>>(part, nslot, out, BH, h0, nh);
  return cudaGetLastError();
}

// ------------------------------------------------------------ copies
__global__ void copy_f32_kernel(float* __restrict__ dst, const float* __restrict__ src,
                                long long n) {
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n;
       i += (long long)gridDim.x * blockDim.x)
    dst[i] = src ? src[i] : 0.f;
}

cudaError_t launch_copy_f32(float* dst, const float* src, long long n, cudaStream_t stream) {
  if (n <= 0) return cudaSuccess;
  long long blocks = (n + 255) / 256;
  if (blocks > 152 * 16) blocks = 152 * 16;
  copy_f32_kernel<<<(int)blocks, 256, 0, stream>>>(dst, src, n);
  return cudaGetLastError();
}

// ------------------------------------------------------------ linear attention
// vt[t, :] = eta[t] * v[t, :] in the work type (bf16: 8 elements per thread).
template <typename T>
__global__ void scale_rows_kernel(const T* __restrict__ v, const float* __restrict__ eta,
                                  T* __restrict__ vt, long long rows, int cols) {
  const long long n = rows * cols;
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n;
       i += (long long)gridDim.x * blockDim.x) {
    const long long r = i / cols;
    vt[i] = from_f<T>(eta[r] * to_f<T>(v[i]));
  }
}

__global__ void scale_rows_bf16x8_kernel(const uint4* __restrict__ v, const float* __restrict__ eta,
                                         uint4* __restrict__ vt, long long n8, int cols8) {
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n8;
       i += (long long)gridDim.x * blockDim.x) {
    const float e = eta[i / cols8];
    uint4 raw = v[i];
    __nv_bfloat162* p = reinterpret_cast<__nv_bfloat162*>(&raw);
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      float2 f = __bfloat1622float2(p[k]);
      p[k] = __floats2bfloat162_rn(e * f.x, e * f.y);
    }
    vt[i] = raw;
  }
}

cudaError_t launch_scale_rows(const void* v, const float* eta, void* vt, long long rows, int cols,
                              bool bf16, cudaStream_t stream) {
  const int threads = 256;
  if (bf16 && cols % 8 == 0) {
    const long long n8 = rows * cols / 8;
    long long blocks = (n8 + threads - 1) / threads;
    if (blocks > 152 * 32) blocks = 152 * 32;
    scale_rows_bf16x8_kernel<<<(int)blocks, threads, 0, stream>>>(
        static_cast<const uint4*>(v), eta, static_cast<uint4*>(vt), n8, cols / 8);
  } else if (bf16) {
    long long blocks = (rows * cols + threads - 1) / threads;
    if (blocks > 152 * 32) blocks = 152 * 32;
    scale_rows_kernel<__nv_bfloat16><<<(int)blocks, threads, 0, stream>>>(
        static_cast<const __nv_bfloat16*>(v), eta, static_cast<__nv_bfloat16*>(vt), rows, cols);
  } else {
    long long blocks = (rows * cols + threads - 1) / threads;
    if (blocks > 152 * 32) blocks = 152 * 32;
    scale_rows_kernel<float><<<(int)blocks, threads, 0, stream>>>(
        static_cast<const float*>(v), eta, static_cast<float*>(vt), rows, cols);
  }
  return cudaGetLastError();
}

// States read by each chunk: S_read[bh, c] = S0 + sum of the partial states of
// the chunks visible to chunk c (earlier chunks for apply-then-update, also
// chunk c otherwise; only flagged chunks in strided mode).  One thread per
// state element and (batch, head), scanning the chunks in order.
template <typename T>
__global__ void linattn_prefix_kernel(const float* __restrict__ partials,
                                      const float* __restrict__ S0, T* __restrict__ s_read,
                                      float* __restrict__ s_final, int BH, int nc, int splits,
                                      int dvdk, int apply_first, UpdateFlags flags) {
  const long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= (long long)BH * dvdk) return;
  const long long bh = i / dvdk;
  const int e = (int)(i - bh * dvdk);
  float s = S0 ? S0[i] : 0.f;
  for (int c = 0; c < nc; ++c) {
    const bool upd = flags.all || ((flags.bits[c >> 5] >> (c & 31)) & 1u);
    float add = 0.f;
    if (upd) {
      const float* p = partials + ((bh * nc + c) * (long long)splits) * dvdk + e;
      for (int sp = 0; sp < splits; ++sp) add += p[(long long)sp * dvdk];
    }
    if (apply_first) {
      s_read[(bh * nc + c) * (long long)dvdk + e] = from_f<T>(s);
      s += add;
    } else {
      s += add;
      s_read[(bh * nc + c) * (long long)dvdk + e] = from_f<T>(s);
    }
  }
  if (s_final) s_final[i] = s;
}

cudaError_t launch_linattn_prefix(const float* partials, const float* S0, void* s_read,
                                  float* s_final, int BH, int nc, int splits, int dvdk,
                                  int apply_first, const UpdateFlags& flags, bool bf16,
                                  cudaStream_t stream) {
  const long long n = (long long)BH * dvdk;
  const int blocks = (int)((n + 255) / 256);
  if (bf16)
    linattn_prefix_kernel<__nv_bfloat16><<<blocks, 256, 0, stream>>>(
        partials, S0, static_cast<__nv_bfloat16*>(s_read), s_final, BH, nc, splits, dvdk,
        apply_first, flags);
  else
    linattn_prefix_kernel<float><<<blocks, 256, 0, stream>>>(
        partials, S0, static_cast<float*>(s_read), s_final, BH, nc, splits, dvdk, apply_first,
        flags);
  return cudaGetLastError();
}

}  // namespace ttt
