// Bandwidth-bound kernels around the GEMMs: fast-weight initialisation and
// operand copies, the update + row L2-normalisation (eq 5/6 of the LaCT
// notes: W <- L2-Normalize(W - U) along the input dimension), the eta
// scaling of linear-attention values, and the prefix of per-chunk
// linear-attention states.
#include "common.cuh"
#include "launch.h"
#include "linattn_kernels.h"

namespace ttt {

// ------------------------------------------------------------ init
// All of a layer call's state setup in one launch: for each of up to three
// weight sets, master = init (broadcast over the batch unless per batch) and
// work = bf16(master); then `nz` floats at `zero` are cleared (momentum,
// squared-norm partials).  Four elements per thread step when every matrix
// size is a multiple of 4 (then all rows are 16-byte aligned).
struct InitArgs {
  MatSet sets[3];
  int nsets, B, H, vec4;
  float* zero[2];
  long long nz[2];
};

__global__ void __launch_bounds__(256) init_layer_kernel(const __grid_constant__ InitArgs a) {
  const long long tid = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  const long long nthreads = (long long)gridDim.x * blockDim.x;
  const int BH = a.B * a.H;
  for (int s = 0; s < a.nsets; ++s) {
    const MatSet& m = a.sets[s];
    const long long per = (long long)m.rows * m.cols;
    __nv_bfloat16* work = static_cast<__nv_bfloat16*>(m.work);
    if (a.vec4) {
      const long long per4 = per / 4, n4 = per4 * BH;
      for (long long i = tid; i < n4; i += nthreads) {
        const long long bh = i / per4, e = i - bh * per4;
        const long long src = (m.init_per_batch ? bh : bh % a.H) * per4 + e;
        const float4 w = reinterpret_cast<const float4*>(m.init)[src];
        reinterpret_cast<float4*>(m.master)[i] = w;
        if (work) {
          __nv_bfloat162 lo = __floats2bfloat162_rn(w.x, w.y), hi = __floats2bfloat162_rn(w.z, w.w);
          uint2 u;
          u.x = *reinterpret_cast<uint32_t*>(&lo);
          u.y = *reinterpret_cast<uint32_t*>(&hi);
          reinterpret_cast<uint2*>(work)[i] = u;
        }
      }
    } else {
      const long long n = per * BH;
      for (long long i = tid; i < n; i += nthreads) {
        const long long bh = i / per, e = i - bh * per;
        const float w = m.init[(m.init_per_batch ? bh : bh % a.H) * per + e];
        m.master[i] = w;
        if (work) work[i] = __float2bfloat16_rn(w);
      }
    }
  }
  for (int z = 0; z < 2; ++z)
    for (long long i = tid; i < a.nz[z]; i += nthreads) a.zero[z][i] = 0.f;
}

cudaError_t launch_init_layer(const MatSet* sets, int nsets, int B, int H, float* zero0,
                              long long n0, float* zero1, long long n1, cudaStream_t stream) {
  InitArgs a{};
  a.nsets = nsets;
  a.B = B;
  a.H = H;
  a.vec4 = 1;
  long long most = 0;
  for (int s = 0; s < nsets; ++s) {
    a.sets[s] = sets[s];
    const long long per = (long long)sets[s].rows * sets[s].cols;
    if (per % 4 != 0) a.vec4 = 0;
    most = per * B * H > most ? per * B * H : most;
  }
  a.zero[0] = zero0;
  a.nz[0] = zero0 ? n0 : 0;
  a.zero[1] = zero1;
  a.nz[1] = zero1 ? n1 : 0;
  most = a.vec4 ? most / 4 : most;
  most = most > a.nz[0] ? most : a.nz[0];
  most = most > a.nz[1] ? most : a.nz[1];
  long long blocks = (most + 255) / 256;
  if (blocks > 152 * 8) blocks = 152 * 8;
  init_layer_kernel<<<(int)(blocks > 0 ? blocks : 1), 256, 0, stream>>>(a);
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
__device__ __forceinline__ bool chunk_flag(const UpdateFlags& f, int c) {
  return f.all || ((f.bits[c >> 5] >> (c & 31)) & 1u);
}

template <typename T>
__global__ void linattn_prefix_kernel(const float* __restrict__ partials,
                                      const float* __restrict__ S0, T* __restrict__ s_read,
                                      float* __restrict__ s_final, int BH, int nc, int splits,
                                      int dvdk, int apply_first, UpdateFlags flags, LinRule rule,
                                      int compact, int n_upd) {
  const long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= (long long)BH * dvdk) return;
  const long long bh = i / dvdk;
  const int e = (int)(i - bh * dvdk);
  float s = S0 ? S0[i] : 0.f;
  float m = rule.M0 ? rule.M0[i] : 0.f;
  int u = 0;
  for (int c = 0; c < nc; ++c) {
    const bool upd = chunk_flag(flags, c);
    float inc = 0.f;
    if (upd) {
      float add = 0.f;
      const float* p = compact ? partials + (bh * n_upd + u) * (long long)dvdk + e
                               : partials + ((bh * nc + c) * (long long)splits) * dvdk + e;
      for (int sp = 0; sp < splits; ++sp) add += p[(long long)sp * dvdk];
      const float lr = (rule.lr ? rule.lr[bh * nc + c] : rule.lr_const) * rule.inc_scale;
      if (rule.mom) {
        m = (rule.alpha ? rule.alpha[bh * nc + c] : rule.alpha_const) * m + add;
        inc = lr * m;
      } else {
        inc = lr * add;
      }
      ++u;
    }
    if (apply_first) {
      s_read[(bh * nc + c) * (long long)dvdk + e] = from_f<T>(s);
      s += inc;
    } else {
      s += inc;
      s_read[(bh * nc + c) * (long long)dvdk + e] = from_f<T>(s);
    }
  }
  if (s_final) s_final[i] = s;
  if (rule.M_final) rule.M_final[i] = m;
}

cudaError_t launch_linattn_prefix(const float* partials, const float* S0, void* s_read,
                                  float* s_final, int BH, int nc, int splits, int dvdk,
                                  int apply_first, const UpdateFlags& flags, const LinRule& rule,
                                  int compact, int n_upd, bool bf16, cudaStream_t stream) {
  const long long n = (long long)BH * dvdk;
  const int blocks = (int)((n + 255) / 256);
  if (bf16)
    linattn_prefix_kernel<__nv_bfloat16><<<blocks, 256, 0, stream>>>(
        partials, S0, static_cast<__nv_bfloat16*>(s_read), s_final, BH, nc, splits, dvdk,
        apply_first, flags, rule, compact, n_upd);
  else
    linattn_prefix_kernel<float><<<blocks, 256, 0, stream>>>(
        partials, S0, static_cast<float*>(s_read), s_final, BH, nc, splits, dvdk, apply_first,
        flags, rule, compact, n_upd);
  return cudaGetLastError();
}

int linattn_momentum_slots(int dvdk) { return (dvdk + 255) / 256; }

// One block = 256 consecutive elements of one batch-head's state; the block's
// squared-norm share of every update is reduced in a fixed order (warp
// shuffles, then the eight warp sums in order).
template <typename T>
__global__ void __launch_bounds__(256)
    linattn_momentum_kernel(const float* __restrict__ partials, int splits, LinRule rule,
                            T* __restrict__ x, float* __restrict__ norm_part, int BH, int nc,
                            int n_upd, int dvdk, UpdateFlags flags) {
  __shared__ float wsum[8];
  const int nslot = (dvdk + 255) / 256;
  const int bh = blockIdx.x / nslot, blk = blockIdx.x % nslot;
  const int e = blk * 256 + threadIdx.x;
  const bool own = e < dvdk;
  const long long i = (long long)bh * dvdk + e;
  float m = (own && rule.M0) ? rule.M0[i] : 0.f;
  int u = 0;
  for (int c = 0; c < nc; ++c) {
    if (!chunk_flag(flags, c)) continue;
    float add = 0.f;
    if (own) {
      const float* p = partials + (((long long)bh * nc + c) * splits) * dvdk + e;
      for (int sp = 0; sp < splits; ++sp) add += p[(long long)sp * dvdk];
      m = (rule.alpha ? rule.alpha[(long long)bh * nc + c] : rule.alpha_const) * m + add;
      x[((long long)bh * n_upd + u) * dvdk + e] = from_f<T>(m);
    }
    float sq = own ? m * m : 0.f;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) sq += __shfl_xor_sync(0xffffffffu, sq, off);
    if ((threadIdx.x & 31) == 0) wsum[threadIdx.x >> 5] = sq;
    __syncthreads();
    if (threadIdx.x == 0) {
      float t = 0.f;
      for (int w = 0; w < 8; ++w) t += wsum[w];
      norm_part[((long long)bh * n_upd + u) * nslot + blk] = t;
    }
    __syncthreads();
    ++u;
  }
  if (own && rule.M_final) rule.M_final[i] = m;
}

cudaError_t launch_linattn_momentum(const float* partials, int splits, const LinRule& rule,
                                    void* x, float* norm_part, int BH, int nc, int n_upd,
                                    int dvdk, const UpdateFlags& flags, bool bf16,
                                    cudaStream_t stream) {
  const int blocks = BH * linattn_momentum_slots(dvdk);
  if (bf16)
    linattn_momentum_kernel<__nv_bfloat16><<<blocks, 256, 0, stream>>>(
        partials, splits, rule, static_cast<__nv_bfloat16*>(x), norm_part, BH, nc, n_upd, dvdk,
        flags);
  else
    linattn_momentum_kernel<float><<<blocks, 256, 0, stream>>>(
        partials, splits, rule, static_cast<float*>(x), norm_part, BH, nc, n_upd, dvdk, flags);
  return cudaGetLastError();
}

__global__ void normsq_sum_kernel(const float* __restrict__ part, int nslot,
                                  float* __restrict__ out, int Z) {
  const int w = (int)((blockIdx.x * blockDim.x + threadIdx.x) >> 5);
  if (w >= Z) return;
  const float s = sum_partials_warp(part + (long long)w * nslot, nslot);
  if ((threadIdx.x & 31) == 0) out[w] = s;
}

cudaError_t launch_normsq_sum(const float* part, int nslot, float* out, int Z,
                              cudaStream_t stream) {
  if (Z <= 0) return cudaSuccess;
  normsq_sum_kernel<<<(Z * 32 + 255) / 256, 256, 0, stream>>>(part, nslot, out, Z);
  return cudaGetLastError();
}

}  // namespace ttt
