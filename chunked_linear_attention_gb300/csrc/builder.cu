#include "builder.h"

#include <cudaTypedefs.h>

#include <cstring>

#include "prof.h"

namespace ttt {

static PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  // looked up once (function-local static initialisation is thread-safe)
  static const PFN_cuTensorMapEncodeTiled_v12000 fn = [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    return static_cast<PFN_cuTensorMapEncodeTiled_v12000>(nullptr);
  }();
  return fn;
}

bool MapCache::get(const TensorRef& t, int box_rows, CUtensorMap* out) {
  for (const Entry& e : entries_)
    if (e.ptr == t.ptr && e.bf16 == t.bf16 && e.rows == t.rows && e.inner == t.inner &&
        e.box_rows == box_rows && e.nblk == 0) {
      *out = e.map;
      return true;
    }
  auto fn = encode_fn();
  if (!fn) return false;
  const int es = t.bf16 ? 2 : 4;
  if ((reinterpret_cast<uintptr_t>(t.ptr) & 15) != 0 || (t.inner * es) % 16 != 0) return false;
  Entry e;
  e.ptr = t.ptr;
  e.bf16 = t.bf16;
  e.rows = t.rows;
  e.inner = t.inner;
  e.box_rows = box_rows;
  e.nblk = 0;
  // one 128-byte swizzle row across: 64 bf16 or 32 fp32 elements
  cuuint64_t dims[2] = {(cuuint64_t)t.inner, (cuuint64_t)t.rows};
  cuuint64_t strides[1] = {(cuuint64_t)t.inner * es};
  cuuint32_t box[2] = {(cuuint32_t)(128 / es), (cuuint32_t)box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(&e.map, t.bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32,
                  2, const_cast<void*>(t.ptr), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return false;
  entries_.push_back(e);
  *out = e.map;
  return true;
}

bool MapCache::get_blocked(const TensorRef& t, int box_rows, int nblk, CUtensorMap* out) {
  for (const Entry& e : entries_)
    if (e.ptr == t.ptr && e.bf16 == t.bf16 && e.rows == t.rows && e.inner == t.inner &&
        e.box_rows == box_rows && e.nblk == nblk) {
      *out = e.map;
      return true;
    }
  auto fn = encode_fn();
  if (!fn || !t.bf16 || nblk < 1 || t.inner % 64 != 0) return false;
  if ((reinterpret_cast<uintptr_t>(t.ptr) & 15) != 0) return false;
  Entry e;
  e.ptr = t.ptr;
  e.bf16 = t.bf16;
  e.rows = t.rows;
  e.inner = t.inner;
  e.box_rows = box_rows;
  e.nblk = nblk;
  cuuint64_t dims[3] = {64, (cuuint64_t)t.rows, (cuuint64_t)(t.inner / 64)};
  cuuint64_t strides[2] = {(cuuint64_t)t.inner * 2, 128};
  cuuint32_t box[3] = {64, (cuuint32_t)box_rows, (cuuint32_t)nblk};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = fn(&e.map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(t.ptr), dims,
                  strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return false;
  entries_.push_back(e);
  *out = e.map;
  return true;
}

LaunchBuilder::LaunchBuilder(bool tensor_cores, MapCache* cache, int* status,
                             unsigned long long wait_ns)
    : tc_(tensor_cores), cache_(cache), ok_(true), status_(status), wait_ns_(wait_ns) {
  reset();
}

void LaunchBuilder::reset() {
  std::memset(&L_, 0, sizeof(L_));
  nmaps_ = 0;
  L_.status = status_;
  L_.wait_limit_ns = wait_ns_;
}

OpDesc LaunchBuilder::op(const TensorRef& t, int mn_major, int outer_base, int z_outer,
                         int box_rows, int mn_krows) {
  OpDesc o;
  std::memset(&o, 0, sizeof(o));
  o.map3 = -1;
  o.mn_major = mn_major;
  o.outer_base = outer_base;
  o.inner_base = 0;
  o.z_outer = z_outer;
  o.z_div = 1;
  const size_t es = t.bf16 ? 2 : 4;
  o.ptr = static_cast<const char*>(t.ptr) + (size_t)outer_base * t.inner * es;
  o.ld = t.inner;
  o.z_stride = (long long)z_outer * t.inner;
  if (tc_) {
    if (!t.bf16) {   // the tensor-core GEMM takes bf16 operands only
      ok_ = false;
      return o;
    }
    const int box = mn_major ? mn_krows : box_rows;
    int slot = -1;
    for (int i = 0; i < nmaps_; ++i)
      if (keys_ptr_[i] == t.ptr && keys_rows_[i] == t.rows && keys_inner_[i] == t.inner &&
          keys_box_[i] == box && keys_nblk_[i] == 0)
        slot = i;
    if (slot < 0) {
      if (nmaps_ >= kMaxMaps || !cache_->get(t, box, &L_.maps[nmaps_])) {
        ok_ = false;
        return o;
      }
      slot = nmaps_++;
      keys_ptr_[slot] = t.ptr;
      keys_rows_[slot] = t.rows;
      keys_inner_[slot] = t.inner;
      keys_box_[slot] = box;
      keys_nblk_[slot] = 0;
    }
    o.map = slot;
    o.map3 = -1;
  }
  return o;
}

int LaunchBuilder::choose_bn(int N, int nacc) const {
  if (!tc_) return kSimtTile;
  // nacc >= 2: bn <= 128 so that accumulators sharing A merge into one N <= 256 MMA
  int max_bn = nacc >= 2 ? 128 : 256;
  int best = 64;
  long long best_area = -1;
  for (int bn = max_bn; bn >= 64; bn -= 64) {
    const long long area = (long long)((N + bn - 1) / bn) * bn;
    if (best_area < 0 || area < best_area) {
      best_area = area;
      best = bn;
    }
  }
  return best;
}

// True if every row the epilogue reads or writes starts on a 32-byte
// boundary: row pitch and batch stride multiples of 16 elements (32 bytes of
// bf16, 64 of fp32) and 32-byte aligned base pointers.
static bool epi_rows32(const EpiDesc& e) {
  if (e.out_ld % 16 != 0 || e.out_z % 16 != 0) return false;
  const void* ptrs[5] = {e.out[0], e.out[1], e.out[2], e.in0, e.mom};
  for (const void* q : ptrs)
    if (q && (reinterpret_cast<uintptr_t>(q) & 31) != 0) return false;
  return true;
}

int LaunchBuilder::blocked_slot(int map2d, int cols) {
  if (map2d < 0 || cols < 128 || cols % 64 != 0 || keys_inner_[map2d] % 64 != 0) return -1;
  const int nblk = cols / 64;
  for (int i = 0; i < nmaps_; ++i)
    if (keys_ptr_[i] == keys_ptr_[map2d] && keys_rows_[i] == keys_rows_[map2d] &&
        keys_inner_[i] == keys_inner_[map2d] && keys_box_[i] == keys_box_[map2d] &&
        keys_nblk_[i] == nblk)
      return i;
  if (nmaps_ >= kMaxMaps) return -1;
  const TensorRef t{keys_ptr_[map2d], 1, keys_rows_[map2d], keys_inner_[map2d]};
  if (!cache_->get_blocked(t, keys_box_[map2d], nblk, &L_.maps[nmaps_])) return -1;
  const int slot = nmaps_++;
  keys_ptr_[slot] = t.ptr;
  keys_rows_[slot] = t.rows;
  keys_inner_[slot] = t.inner;
  keys_box_[slot] = keys_box_[map2d];
  keys_nblk_[slot] = nblk;
  return slot;
}

bool LaunchBuilder::add(Problem p) {
  if (L_.nprob >= kMaxProblems) {
    ok_ = false;
    return false;
  }
  p.epi.rows32 = epi_rows32(p.epi) ? 1 : 0;
  if (tc_ && p.kd == 2) {   // two K steps per stage: one accumulator, K % 128, MN-major boxes
    bool good = p.K % 128 == 0 && p.nacc == 1;   // 128 K rows deep
    for (int j = 0; j < p.nacc; ++j) {
      if (p.a[j].mn_major && keys_box_[p.a[j].map] != 128) good = false;
      if (p.b[j].mn_major && keys_box_[p.b[j].map] != 128) good = false;
    }
    if (!good) {
      ok_ = false;
      return false;
    }
  }
  if (!tc_) p.kd = 1;
  if (tc_) {
    // MN-major tiles of two or more 64-column blocks: one 3-D box per stage
    // instead of one box per block (fewer, larger TMA transfers)
    for (int j = 0; j < p.nacc; ++j) {
      if (p.a[j].mn_major && p.a[j].inner_base % 64 == 0)
        p.a[j].map3 = blocked_slot(p.a[j].map, bm());
      if (p.b[j].mn_major && p.b[j].inner_base % 64 == 0)
        p.b[j].map3 = blocked_slot(p.b[j].map, p.bn);
    }
  }
  const int bm = this->bm();
  if (!tc_) p.bn = kSimtTile;
  p.tiles_m = (p.M + bm - 1) / bm;
  p.tiles_n = (p.N + p.bn - 1) / p.bn;
  p.tile_start = L_.total_tiles;
  L_.prob[L_.nprob++] = p;
  L_.total_tiles += p.tiles_m * p.tiles_n * p.Z;
  return true;
}

cudaError_t LaunchBuilder::launch(cudaStream_t stream, int tag, int priority, int max_ctas) {
  if (!ok_) return cudaErrorInvalidValue;
  double flops = 0;
  for (int i = 0; i < L_.nprob; ++i) {
    const Problem& p = L_.prob[i];
    flops += 2.0 * p.M * p.N * (double)p.K * p.Z * p.nacc;
  }
  cudaError_t e;
  {
    const int sms = tc_ ? device_sm_count() : 0;
    const double share = sms > 0 ? (double)umma_gemm_grid(L_, max_ctas) / sms : 1.0;
    ProfScope ps(tag, stream, flops, 0.0, share);
    e = tc_ ? launch_umma_gemm(L_, stream, priority, max_ctas) : launch_simt_gemm(L_, stream);
  }
  reset();
  return e;
}

}  // namespace ttt
