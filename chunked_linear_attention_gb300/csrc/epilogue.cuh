// Fused GEMM epilogues.  Each call handles V consecutive output columns of one
// output row (one token, or one row of a fast-weight matrix) and receives the
// matching accumulator values of up to three accumulators.
//
//   EPI_PROJ_Q   A_q = SiLU(H1) * H3                         (eq 3, queries)
//                times -eta of the row when eta is given (P of a static
//                feature map), or the constant a when a != 0
//   EPI_PROJ_K   dA = -eta * (V W2);  s = sigmoid(H1)
//                dH1 = dA * H3 * s (1 + H1 (1 - s))  (SiLU', App. I.1)
//                dH3 = dA * SiLU(H1);  P = -eta * SiLU(H1) * H3
//                so that g1 = dH1^T K, g3 = dH3^T K, g2 = V^T P (eqs 2, 4)
//   EPI_GRAD     M = beta M + g (momentum sentence after eq 6); then the
//                update source U = M (fp32) or the Newton-Schulz input X = M
//                (work type) with its squared Frobenius norm accumulated
//   EPI_OUT      o = acc (layer output, I/O type)
//   EPI_NS_GRAM  A = s^2 X X^T,     s = 1/(|M|_F + eps) on the first step
//   EPI_NS_POLY  B = b A + c A A
//   EPI_NS_STEP  X' = s (a X + B X)  (work type, or fp32 U on the last step)
//
// All packing is done in registers (no address-taken local arrays), so the
// epilogue never touches local memory.
#pragma once

#include "common.cuh"

namespace ttt {

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}
__device__ __forceinline__ float bf16lo(uint32_t x) { return __uint_as_float(x << 16); }
__device__ __forceinline__ float bf16hi(uint32_t x) { return __uint_as_float(x & 0xffff0000u); }

// Stores V values; vector path when all V are valid and dst is 16-byte aligned.
template <typename T, int V>
__device__ __forceinline__ void store_vec(T* dst, const float (&v)[V], int n) {
  if constexpr (sizeof(T) == 2) {
    if (V % 8 == 0 && n == V && (reinterpret_cast<uintptr_t>(dst) & 15) == 0) {
#pragma unroll
      for (int i = 0; i < V; i += 8)
        *reinterpret_cast<uint4*>(dst + i) =
            make_uint4(pack_bf16x2(v[i], v[i + 1]), pack_bf16x2(v[i + 2], v[i + 3]),
                       pack_bf16x2(v[i + 4], v[i + 5]), pack_bf16x2(v[i + 6], v[i + 7]));
      return;
    }
  } else {
    if (V % 4 == 0 && n == V && (reinterpret_cast<uintptr_t>(dst) & 15) == 0) {
#pragma unroll
      for (int i = 0; i < V; i += 4)
        *reinterpret_cast<float4*>(dst + i) = make_float4(v[i], v[i + 1], v[i + 2], v[i + 3]);
      return;
    }
  }
#pragma unroll
  for (int i = 0; i < V; ++i)
    if (i < n) dst[i] = from_f<T>(v[i]);
}

template <typename T, int V>
__device__ __forceinline__ void load_vec(const T* src, float (&v)[V], int n) {
  if constexpr (sizeof(T) == 2) {
    if (V % 8 == 0 && n == V && (reinterpret_cast<uintptr_t>(src) & 15) == 0) {
#pragma unroll
      for (int i = 0; i < V; i += 8) {
        const uint4 r = *reinterpret_cast<const uint4*>(src + i);
        v[i] = bf16lo(r.x); v[i + 1] = bf16hi(r.x);
        v[i + 2] = bf16lo(r.y); v[i + 3] = bf16hi(r.y);
        v[i + 4] = bf16lo(r.z); v[i + 5] = bf16hi(r.z);
        v[i + 6] = bf16lo(r.w); v[i + 7] = bf16hi(r.w);
      }
      return;
    }
  } else {
    if (V % 4 == 0 && n == V && (reinterpret_cast<uintptr_t>(src) & 15) == 0) {
#pragma unroll
      for (int i = 0; i < V; i += 4) {
        const float4 f = *reinterpret_cast<const float4*>(src + i);
        v[i] = f.x; v[i + 1] = f.y; v[i + 2] = f.z; v[i + 3] = f.w;
      }
      return;
    }
  }
#pragma unroll
  for (int i = 0; i < V; ++i) v[i] = i < n ? to_f<T>(src[i]) : 0.f;
}

// 1 / (|M|_F + eps) from an accumulated squared norm.
__device__ __forceinline__ float ns_scale(const EpiDesc& e, int z) {
  return 1.0f / (sqrtf(e.normsq[z]) + e.eps);
}

// WT: work tensors (bf16 on the tensor-core path, fp32 on the SIMT path).
// IOT: layer input/output type.  `r` is the row inside the problem's M range,
// `c` the first of the n (<= V) valid columns.  Returns the sum of squares
// of the values EPI_GRAD routes to the Newton-Schulz input (else 0).
template <int V, typename WT, typename IOT, bool kPrecise>
__device__ __forceinline__ float epilogue_vec(const EpiDesc& e, int z, int r, int c, int n,
                                              const float (&a0)[V], const float (&a1)[V],
                                              const float (&a2)[V]) {
  const int zz = e.z_div > 1 ? z / e.z_div : z;
  const long long idx = (long long)zz * e.out_z + (e.out_row0 + r) * e.out_ld + c;
  float o[V];
  float sumsq = 0.f;
  switch (e.kind) {
    case EPI_STORE_F32: {
      store_vec<float, V>(static_cast<float*>(e.out[0]) + idx, a0, n);
      break;
    }
    case EPI_PROJ_Q: {
      // optional row factor: -eta of the row (e.eta set) or the constant e.a
      const float f = e.eta ? -e.eta[(long long)zz * e.eta_z + e.eta_row0 + r]
                            : (e.a != 0.f ? e.a : 1.0f);
#pragma unroll
      for (int i = 0; i < V; ++i) {
        const float s = kPrecise ? sigmoid_precise(a0[i]) : sigmoid_f(a0[i]);
        o[i] = a0[i] * s * a1[i] * f;
      }
      store_vec<WT, V>(static_cast<WT*>(e.out[0]) + idx, o, n);
      break;
    }
    case EPI_PROJ_K: {
      const float eta = e.eta[(long long)zz * e.eta_z + e.eta_row0 + r];
      float dh1[V], dh3[V];
#pragma unroll
      for (int i = 0; i < V; ++i) {
        const float h1 = a0[i], h3 = a1[i];
        const float s = kPrecise ? sigmoid_precise(h1) : sigmoid_f(h1);
        const float sl = h1 * s;
        const float dA = -eta * a2[i];
        dh1[i] = dA * h3 * s * (1.0f + h1 * (1.0f - s));
        dh3[i] = dA * sl;
        o[i] = -eta * sl * h3;
      }
      store_vec<WT, V>(static_cast<WT*>(e.out[0]) + idx, dh1, n);
      store_vec<WT, V>(static_cast<WT*>(e.out[1]) + idx, dh3, n);
      store_vec<WT, V>(static_cast<WT*>(e.out[2]) + idx, o, n);
      break;
    }
    case EPI_GRAD: {
      if (e.mom) {
        float m[V];
        load_vec<float, V>(e.mom + idx, m, n);
#pragma unroll
        for (int i = 0; i < V; ++i) o[i] = e.a * m[i] + a0[i];
        store_vec<float, V>(e.mom + idx, o, n);
      } else {
#pragma unroll
        for (int i = 0; i < V; ++i) o[i] = a0[i];
      }
      if (e.out[0]) store_vec<float, V>(static_cast<float*>(e.out[0]) + idx, o, n);
      if (e.out[1]) {
        store_vec<WT, V>(static_cast<WT*>(e.out[1]) + idx, o, n);
#pragma unroll
        for (int i = 0; i < V; ++i)
          if (i < n) sumsq += o[i] * o[i];
      }
      break;
    }
    case EPI_OUT: {
      store_vec<IOT, V>(static_cast<IOT*>(e.out[0]) + idx, a0, n);
      break;
    }
    case EPI_NS_GRAM: {
      const float s = e.first ? ns_scale(e, zz) : 1.0f;
      const float s2 = s * s;
#pragma unroll
      for (int i = 0; i < V; ++i) o[i] = a0[i] * s2;
      store_vec<WT, V>(static_cast<WT*>(e.out[0]) + idx, o, n);
      break;
    }
    case EPI_NS_POLY: {
      float x[V];
      load_vec<WT, V>(static_cast<const WT*>(e.in0) + idx, x, n);
#pragma unroll
      for (int i = 0; i < V; ++i) o[i] = e.b * x[i] + e.c * a0[i];
      store_vec<WT, V>(static_cast<WT*>(e.out[0]) + idx, o, n);
      break;
    }
    case EPI_NS_STEP: {
      const float s = e.first ? ns_scale(e, zz) : 1.0f;
      float x[V];
      load_vec<WT, V>(static_cast<const WT*>(e.in0) + idx, x, n);
#pragma unroll
      for (int i = 0; i < V; ++i) o[i] = s * (e.a * x[i] + a0[i]);
      if (e.out[1])
        store_vec<float, V>(static_cast<float*>(e.out[1]) + idx, o, n);
      else
        store_vec<WT, V>(static_cast<WT*>(e.out[0]) + idx, o, n);
      break;
    }
    default:
      break;
  }
  return sumsq;
}

}  // namespace ttt
