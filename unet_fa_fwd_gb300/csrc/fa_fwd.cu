// fa_fwd.cu — C ABI of the attention forward (declared in include/fa.h):
// argument validation, TMA descriptor encoding and the kernel launches.  The
// attention kernel itself is compiled per head dimension in
// fa_attn_d{32,64,128}.cu (see fa_attn_launch.h).
//
// The library is linked against the static CUDA runtime and reaches the
// driver's tensor-map encoder through cudaGetDriverEntryPointByVersion, so it
// loads on a machine without a GPU driver; every compute entry point then
// fails with FA_ERR_CUDA instead of crashing.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <climits>
#include <cmath>
#include <cstdarg>
#include <cstdint>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>

#include "fa.h"
#include "fa_attn_launch.h"
#include "fa_log.h"
#include "fa_quant.cuh"
#include "fa_window_geom.h"
#include "fa_diag.cuh"

// Device status word (one per device): 0, or FA_ERR_TIMEOUT once a kernel
// wait ran out of time.  Kernels in every translation unit receive its device
// address in their parameters.
__device__ int g_device_status = 0;
// First failed device-side check of a debug build (see fa_debug_report).
__device__ int g_debug_record[8] = {};

namespace {

constexpr int kMaxDevices = 64;

struct DeviceState {
  bool ready = false;
  bool supported = false;
  int device = 0;
  int sm_count = 0;
  int* status = nullptr;  // device address of g_device_status
  int* debug_record = nullptr;  // device address of g_debug_record
};

std::mutex g_mutex;
DeviceState g_devices[kMaxDevices];
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

bool ranges_overlap(const void* a, size_t abytes, const void* b, size_t bbytes) {
  if (!a || !b || abytes == 0 || bbytes == 0) return false;
  const uintptr_t a0 = reinterpret_cast<uintptr_t>(a), b0 = reinterpret_cast<uintptr_t>(b);
  return a0 < b0 + bbytes && b0 < a0 + abytes;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

unsigned long long timeout_ns_from_env() {
  const char* e = std::getenv("FA_WAIT_TIMEOUT_MS");
  if (e && *e) {
    char* end = nullptr;
    unsigned long long ms = std::strtoull(e, &end, 10);
    if (end != e && ms > 0) return ms * 1000000ull;
  }
  return 2000ull * 1000000ull;  // 2 s per wait; a healthy wait lasts microseconds
}

// Set-up per device: capability check, SM count, driver entry point.
int device_setup(int dev, DeviceState** out) {
  if (dev < 0 || dev >= kMaxDevices) return FA_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_mutex);
  DeviceState& st = g_devices[dev];
  if (!st.ready) {
    int major = 0, minor = 0, sms = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
      return FA_ERR_CUDA;
    }
    st.supported = (major == 10 && minor == 3);
    st.device = dev;
    st.sm_count = sms;
    void* status = nullptr;
    if (cudaGetSymbolAddress(&status, g_device_status) != cudaSuccess || !status) return FA_ERR_CUDA;
    st.status = static_cast<int*>(status);
    void* rec = nullptr;
    if (cudaGetSymbolAddress(&rec, g_debug_record) != cudaSuccess || !rec) return FA_ERR_CUDA;
    st.debug_record = static_cast<int*>(rec);
    if (!g_encode) {
      void* fn = nullptr;
      cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
      if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                           &q) != cudaSuccess ||
          q != cudaDriverEntryPointSuccess || fn == nullptr) {
        return FA_ERR_CUDA;
      }
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    }
    st.ready = true;
  }
  *out = &st;
  return FA_OK;
}

// 3-D tensor map over a contiguous bf16 [BH][N][D] tensor; box = one chunk of
// 128 rows (inner extent = the swizzle span), swizzled to match the UMMA
// shared-memory layout.
int encode_map(CUtensorMap* map, const void* base, int BH, int N, int D) {
  const int sw_bytes = (D >= 64) ? 128 : 64;
  cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)N, (cuuint64_t)BH};
  cuuint64_t strides[2] = {(cuuint64_t)D * 2, (cuuint64_t)N * D * 2};
  cuuint32_t box[3] = {(cuuint32_t)(sw_bytes / 2), 128u, 1u};
  cuuint32_t estride[3] = {1u, 1u, 1u};
  CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims,
                        strides, box, estride, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        sw_bytes == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? FA_OK : FA_ERR_CUDA;
}

// 4-D tensor map over a per-(query, key) fp32 mask [B][heads][Nq][Nk] (Nk a
// multiple of 4).  Box = 128 query rows x 32 keys (128 bytes), 128-byte
// swizzle.  Coordinates past Nq or Nk read zeros (those rows and keys are
// never used).
int encode_mask_map(CUtensorMap* map, const void* base, int B, int heads, int Nq, int Nk) {
  cuuint64_t dims[4] = {(cuuint64_t)Nk, (cuuint64_t)Nq, (cuuint64_t)heads, (cuuint64_t)B};
  cuuint64_t strides[3] = {(cuuint64_t)Nk * 4, (cuuint64_t)Nq * Nk * 4,
                           (cuuint64_t)heads * Nq * Nk * 4};
  cuuint32_t box[4] = {32u, 128u, 1u, 1u};
  cuuint32_t estride[4] = {1u, 1u, 1u, 1u};
  CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32,
                        4, const_cast<void*>(base), dims, strides, box, estride,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? FA_OK : FA_ERR_CUDA;
}

int launch_merge(const float* part_o, const float* part_lse, __nv_bfloat16* out, float* lse,
                 int splits, long long rows, int D, cudaStream_t s) {
  const int rows_per_block = 256 / 32;
  const long long blocks = (rows + rows_per_block - 1) / rows_per_block;
  if (blocks > INT_MAX) return FA_ERR_INVALID_ARGUMENT;
  fa::log_launch("fa_merge_kernel<D=%d> grid %lld x 256 threads, %d ranges, %lld rows", D, blocks,
             splits, rows);
  switch (D) {
    case 32: fa::fa_merge_kernel<32><<<(int)blocks, 256, 0, s>>>(part_o, part_lse, out, lse, splits, rows); break;
    case 64: fa::fa_merge_kernel<64><<<(int)blocks, 256, 0, s>>>(part_o, part_lse, out, lse, splits, rows); break;
    default: fa::fa_merge_kernel<128><<<(int)blocks, 256, 0, s>>>(part_o, part_lse, out, lse, splits, rows); break;
  }
  return cudaGetLastError() == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

// Sizes of one validated problem (no CUDA call was needed to get them).
struct Shape {
  int64_t BH, upb;
  size_t q_bytes, kv_bytes, lse_bytes, mask_bytes;
};

// Validation shared by the entry points; makes no CUDA call, so an invalid
// call returns before anything touches the device.
int validate(const void* q, const void* k, const void* v, const float* mask, const void* out,
             const float* lse, int B, int H, int Nq, int Nk, int D, float scale, Shape* sh) {
  if (!q || !k || !v || !out || !lse) return FA_ERR_INVALID_ARGUMENT;
  if (B < 1 || H < 1 || Nq < 1 || Nk < 1) return FA_ERR_INVALID_ARGUMENT;
  if (!std::isfinite(scale)) return FA_ERR_INVALID_ARGUMENT;
  if (D != 32 && D != 64 && D != 128) return FA_ERR_UNSUPPORTED;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out) || !aligned16(lse) ||
      (mask && !aligned16(mask)))
    return FA_ERR_INVALID_ARGUMENT;
  const int64_t BH = (int64_t)B * H;
  const int64_t qtiles = ((int64_t)Nq + 127) / 128;
  const int64_t upb = (qtiles + 1) / 2;
  if (BH > INT_MAX || BH * upb > INT_MAX || BH > (int64_t)UINT32_MAX) return FA_ERR_INVALID_ARGUMENT;
  sh->BH = BH;
  sh->upb = upb;
  sh->q_bytes = (size_t)BH * Nq * D * 2;
  sh->kv_bytes = (size_t)BH * Nk * D * 2;
  sh->lse_bytes = (size_t)BH * Nq * 4;
  sh->mask_bytes = mask ? (size_t)B * Nk * 4 : 0;
  const size_t qb = sh->q_bytes, kvb = sh->kv_bytes, lb = sh->lse_bytes, mb = sh->mask_bytes;
  if (ranges_overlap(out, qb, q, qb) || ranges_overlap(out, qb, k, kvb) ||
      ranges_overlap(out, qb, v, kvb) || ranges_overlap(out, qb, lse, lb) ||
      ranges_overlap(out, qb, mask, mb) || ranges_overlap(lse, lb, q, qb) ||
      ranges_overlap(lse, lb, k, kvb) || ranges_overlap(lse, lb, v, kvb) ||
      ranges_overlap(lse, lb, mask, mb))
    return FA_ERR_INVALID_ARGUMENT;
  return FA_OK;
}

// A workspace must not overlap any buffer of the call.
bool workspace_overlaps(const void* ws, size_t ws_bytes, const void* q, const void* k,
                        const void* v, const float* mask, const void* out, const float* lse,
                        const Shape& sh) {
  return ranges_overlap(ws, ws_bytes, q, sh.q_bytes) || ranges_overlap(ws, ws_bytes, k, sh.kv_bytes) ||
         ranges_overlap(ws, ws_bytes, v, sh.kv_bytes) || ranges_overlap(ws, ws_bytes, out, sh.q_bytes) ||
         ranges_overlap(ws, ws_bytes, lse, sh.lse_bytes) ||
         ranges_overlap(ws, ws_bytes, mask, sh.mask_bytes);
}

// Set-up of a validated call (CUDA calls, nothing enqueued): device state and
// the tensor maps and sizes of an unsplit launch.
int setup(const void* q, const void* k, const void* v, const float* mask, void* out, float* lse,
          int H, int Nq, int Nk, int D, float scale, const Shape& sh, fa::Params* prm,
          DeviceState** st) {
  const char* inject = std::getenv("FA_FAULT_INJECT");
  if (inject && std::strcmp(inject, "launch") == 0) return FA_ERR_CUDA;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return FA_ERR_CUDA;
  int rc = device_setup(dev, st);
  if (rc != FA_OK) return rc;
  if (!(*st)->supported) return FA_ERR_UNSUPPORTED;

  std::memset(prm, 0, sizeof(*prm));
  if (encode_map(&prm->tm_q, q, (int)sh.BH, Nq, D) != FA_OK ||
      encode_map(&prm->tm_k, k, (int)sh.BH, Nk, D) != FA_OK ||
      encode_map(&prm->tm_v, v, (int)sh.BH, Nk, D) != FA_OK)
    return FA_ERR_CUDA;
  prm->out = reinterpret_cast<__nv_bfloat16*>(out);
  prm->lse = lse;
  prm->mask = mask;
  // A key-padding row is read 16 bytes at a time when every batch row starts
  // 16-byte aligned (the base is, so Nk % 4 == 0 suffices).
  prm->mask_kind = mask ? ((Nk % 4 == 0) ? fa::kMaskF32Vec : fa::kMaskF32Scalar) : fa::kMaskNone;
  prm->H = H;
  prm->Nq = Nq;
  prm->Nk = Nk;
  prm->BH = (int)sh.BH;
  prm->units_per_bh = (int)sh.upb;
  prm->nkv = (Nk + 127) / 128;
  prm->num_splits = 1;
  prm->mask_heads = 1;
  prm->num_units = (int)(sh.BH * sh.upb);
  prm->div_upb = fa::FastDiv::make((uint32_t)sh.upb);
  prm->div_splits = fa::FastDiv::make(1);
  prm->div_bh = fa::FastDiv::make((uint32_t)sh.BH);
  prm->div_h = fa::FastDiv::make((uint32_t)H);
  prm->scale_log2 = (float)((double)scale * 1.4426950408889634);
  prm->timeout_ns = timeout_ns_from_env();
  prm->status = (*st)->status;
  prm->debug_record = (*st)->debug_record;
#ifdef FA_DEBUG
  const char* plant = std::getenv("FA_DEBUG_PLANT");
  prm->debug_plant = (plant && std::strcmp(plant, "store") == 0) ? 1 : 0;
#endif
  prm->inject_stall = (inject && std::strcmp(inject, "stall") == 0) ? 1 : 0;
  return FA_OK;
}

int launch_fwd(const fa::Params& prm_in, DeviceState& st, int D, cudaStream_t s, bool f8 = false) {
  fa::Params prm = prm_in;
  fa::plan_last_wave(prm, st.sm_count);
  switch (D) {
    case 32: return fa::launch_attention_d32(prm, f8, st.device, st.sm_count, s);
    case 64: return fa::launch_attention_d64(prm, f8, st.device, st.sm_count, s);
    default: return fa::launch_attention_d128(prm, f8, st.device, st.sm_count, s);
  }
}

// 3-D tensor map over a contiguous e4m3 [BH][N][D] tensor: one box row is the
// whole D-byte row, swizzled over D bytes (128 / 64 / 32).
int encode_map_f8(CUtensorMap* map, const void* base, int BH, int N, int D) {
  cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)N, (cuuint64_t)BH};
  cuuint64_t strides[2] = {(cuuint64_t)D, (cuuint64_t)N * D};
  cuuint32_t box[3] = {(cuuint32_t)D, 128u, 1u};
  cuuint32_t estride[3] = {1u, 1u, 1u};
  const CUtensorMapSwizzle sw = D == 128 ? CU_TENSOR_MAP_SWIZZLE_128B
                                         : (D == 64 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_32B);
  CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(base), dims, strides,
                        box, estride, CU_TENSOR_MAP_INTERLEAVE_NONE, sw,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? FA_OK : FA_ERR_CUDA;
}

// Workspace of the FP8 forward, in order (each part 256-byte aligned).
struct F8Layout {
  size_t q8, k8, q_scale, k_scale, mean, partial, corr, total;
};
constexpr int kF8ColsumSplits = 64;

F8Layout f8_layout(int B, int H, int Nq, int Nk, int D) {
  const size_t BH = (size_t)B * H;
  const size_t qt = ((size_t)Nq + 127) / 128, kt = ((size_t)Nk + 127) / 128;
  F8Layout l{};
  size_t off = 0;
  l.q8 = off;       off += align256(BH * Nq * D);
  l.k8 = off;       off += align256(BH * Nk * D);
  l.q_scale = off;  off += align256(BH * qt * 4);
  l.k_scale = off;  off += align256(BH * kt * 4);
  l.mean = off;     off += align256(BH * D * 4);
  l.partial = off;  off += align256(BH * kF8ColsumSplits * D * 4);
  l.corr = off;     off += align256(BH * Nq * 4);
  l.total = off;
  return l;
}

template <int D>
void launch_quant(const void* q, const void* k, char* ws, const F8Layout& L, int BH, int Nq, int Nk,
                  float scale, cudaStream_t s) {
  const int kt = (Nk + 127) / 128, qt = (Nq + 127) / 128;
  fa::log_launch("fa_k_colsum_kernel<D=%d> grid %d x %d; fa_k_mean_kernel grid %d; "
                 "fa_quant_kernel<D=%d> grid %d (%d K blocks + %d Q blocks; 256 threads each)",
                 D, BH, kF8ColsumSplits, (BH * D + 255) / 256, D, BH * (kt + qt), BH * kt, BH * qt);
  fa::fa_k_colsum_kernel<D><<<dim3(BH, kF8ColsumSplits), 256, 0, s>>>(
      static_cast<const __nv_bfloat16*>(k), reinterpret_cast<float*>(ws + L.partial), Nk,
      kF8ColsumSplits);
  fa::fa_k_mean_kernel<<<(BH * D + 255) / 256, 256, 0, s>>>(
      reinterpret_cast<const float*>(ws + L.partial), reinterpret_cast<float*>(ws + L.mean), BH, D,
      kF8ColsumSplits, Nk);
  fa::fa_quant_kernel<D><<<BH * (kt + qt), 256, 0, s>>>(
      static_cast<const __nv_bfloat16*>(k), static_cast<const __nv_bfloat16*>(q),
      reinterpret_cast<const float*>(ws + L.mean),
      reinterpret_cast<uint8_t*>(ws + L.k8), reinterpret_cast<uint8_t*>(ws + L.q8),
      reinterpret_cast<float*>(ws + L.k_scale), reinterpret_cast<float*>(ws + L.q_scale),
      reinterpret_cast<float*>(ws + L.corr), BH, Nk, Nq, kt, qt, scale);
}

// Key ranges actually used for a requested count: at most one per key block,
// so that every range is non-empty.
int effective_splits(int nkv, int requested) { return requested < nkv ? requested : nkv; }


}  // namespace

// Fixed scratch of fa_fwd_split_noalloc (file scope, internal linkage): every
// GPU that loads the library holds it until the process exits.  Host code
// must not pass its name to a kernel (it is a host-side stand-in); the device
// address comes from cudaGetSymbolAddress, cached per device.
static __device__ __align__(256) unsigned char g_noalloc_scratch[FA_NOALLOC_SCRATCH_BYTES];
static void* g_noalloc_scratch_addr[kMaxDevices] = {};

extern "C" {

int fa_fwd(const void* q, const void* k, const void* v, const float* mask, void* out, float* lse,
           int B, int H, int Nq, int Nk, int D, float scale, void* stream) {
  Shape sh;
  int rc = validate(q, k, v, mask, out, lse, B, H, Nq, Nk, D, scale, &sh);
  if (rc != FA_OK) return rc;
  fa::Params prm;
  DeviceState* st = nullptr;
  rc = setup(q, k, v, mask, out, lse, H, Nq, Nk, D, scale, sh, &prm, &st);
  if (rc != FA_OK) return rc;
  return launch_fwd(prm, *st, D, reinterpret_cast<cudaStream_t>(stream));
}

int fa_fwd_ex(const void* q, const void* k, const void* v, const fa_mask* mask, int causal,
              void* out, float* lse, int B, int H, int Nq, int Nk, int D, float scale,
              void* stream) {
  const int kind = mask ? mask->kind : FA_MASK_NONE;
  if (kind != FA_MASK_NONE && kind != FA_MASK_KEY_PADDING && kind != FA_MASK_ADDITIVE &&
      kind != FA_MASK_BOOL)
    return FA_ERR_INVALID_ARGUMENT;
  if (kind != FA_MASK_NONE && !mask->data) return FA_ERR_INVALID_ARGUMENT;
  const bool full = kind == FA_MASK_ADDITIVE || kind == FA_MASK_BOOL;
  if (full) {
    if (mask->heads != 1 && mask->heads != H) return FA_ERR_INVALID_ARGUMENT;
    if (kind == FA_MASK_ADDITIVE && (reinterpret_cast<uintptr_t>(mask->data) & 3u))
      return FA_ERR_INVALID_ARGUMENT;
  }
  const float* key_mask = kind == FA_MASK_KEY_PADDING ? static_cast<const float*>(mask->data) : nullptr;
  Shape sh;
  int rc = validate(q, k, v, key_mask, out, lse, B, H, Nq, Nk, D, scale, &sh);
  if (rc != FA_OK) return rc;
  if (full) {
    const size_t fm_bytes =
        (size_t)B * mask->heads * Nq * Nk * (kind == FA_MASK_ADDITIVE ? sizeof(float) : 1);
    if (ranges_overlap(mask->data, fm_bytes, out, sh.q_bytes) ||
        ranges_overlap(mask->data, fm_bytes, lse, sh.lse_bytes))
      return FA_ERR_INVALID_ARGUMENT;
  }
  fa::Params prm;
  DeviceState* st = nullptr;
  rc = setup(q, k, v, key_mask, out, lse, H, Nq, Nk, D, scale, sh, &prm, &st);
  if (rc != FA_OK) return rc;
  if (full) {
    prm.full_mask = mask->data;
    prm.full_mask_bool = kind == FA_MASK_BOOL;
    prm.mask_heads = mask->heads;
    // When every mask row starts 16-byte aligned (Nk * element size a
    // multiple of 16 and an aligned base), an fp32 mask is staged (copied by
    // TMA into shared memory tile by tile; 1.7x faster than 16-byte loads of
    // each row on FLUX 1024) and a byte mask is read with 16-byte loads (a
    // quarter of the traffic: its plain loads measured faster than staging
    // it, which costs K/V ring depth); otherwise each lane reads its row
    // element by element.
    const bool bytes = kind == FA_MASK_BOOL;
    const bool rows16 = aligned16(mask->data) && Nk % (bytes ? 16 : 4) == 0;
    if (bytes) {
      prm.mask_kind = rows16 ? fa::kMaskU8Vec : fa::kMaskU8Scalar;
    } else if (rows16) {
      if (encode_mask_map(&prm.tm_mask, mask->data, B, mask->heads, Nq, Nk) != FA_OK)
        return FA_ERR_CUDA;
      prm.mask_kind = fa::kMaskF32Staged;
    } else {
      prm.mask_kind = fa::kMaskF32Scalar;
    }
  }
  prm.causal = causal ? 1 : 0;
  return launch_fwd(prm, *st, D, reinterpret_cast<cudaStream_t>(stream));
}

size_t fa_fp8_workspace_bytes(int B, int H, int Nq, int Nk, int D) {
  if (B < 1 || H < 1 || Nq < 1 || Nk < 1 || (D != 32 && D != 64 && D != 128)) return 0;
  return f8_layout(B, H, Nq, Nk, D).total;
}

int fa_fwd_fp8(const void* q, const void* k, const void* v, const float* mask, void* out,
               float* lse, int B, int H, int Nq, int Nk, int D, float scale, void* workspace,
               size_t workspace_bytes, void* stream) {
  Shape sh;
  int rc = validate(q, k, v, mask, out, lse, B, H, Nq, Nk, D, scale, &sh);
  if (rc != FA_OK) return rc;
  if (!workspace || !aligned16(workspace)) return FA_ERR_INVALID_ARGUMENT;
  const F8Layout L = f8_layout(B, H, Nq, Nk, D);
  if (workspace_bytes < L.total) return FA_ERR_INVALID_ARGUMENT;
  if (workspace_overlaps(workspace, L.total, q, k, v, mask, out, lse, sh))
    return FA_ERR_INVALID_ARGUMENT;
  fa::Params prm;
  DeviceState* st = nullptr;
  rc = setup(q, k, v, mask, out, lse, H, Nq, Nk, D, scale, sh, &prm, &st);
  if (rc != FA_OK) return rc;
  char* ws = static_cast<char*>(workspace);
  if (encode_map_f8(&prm.tm_q, ws + L.q8, prm.BH, Nq, D) != FA_OK ||
      encode_map_f8(&prm.tm_k, ws + L.k8, prm.BH, Nk, D) != FA_OK)
    return FA_ERR_CUDA;
  prm.q_scale = reinterpret_cast<const float*>(ws + L.q_scale);
  prm.k_scale = reinterpret_cast<const float*>(ws + L.k_scale);
  prm.lse_corr = reinterpret_cast<const float*>(ws + L.corr);
  prm.qtiles = (Nq + 127) / 128;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  switch (D) {
    case 32: launch_quant<32>(q, k, ws, L, prm.BH, Nq, Nk, scale, s); break;
    case 64: launch_quant<64>(q, k, ws, L, prm.BH, Nq, Nk, scale, s); break;
    default: launch_quant<128>(q, k, ws, L, prm.BH, Nq, Nk, scale, s); break;
  }
  if (cudaGetLastError() != cudaSuccess) return FA_ERR_CUDA;
  return launch_fwd(prm, *st, D, s, true);
}

size_t fa_split_workspace_bytes(int B, int H, int Nq, int D, int num_splits) {
  if (B < 1 || H < 1 || Nq < 1 || D < 1 || num_splits < 1) return 0;
  const size_t rows = (size_t)B * H * Nq * num_splits;
  return align256(rows * D * sizeof(float)) + align256(rows * sizeof(float));
}

int fa_split_count(int B, int H, int Nq, int Nk, int num_sms) {
  if (B < 1 || H < 1 || Nq < 1 || Nk < 1 || num_sms < 1) return 1;
  const long long units = (long long)B * H * ((((long long)Nq + 127) / 128 + 1) / 2);
  const int nkv = (Nk + 127) / 128;
  if (units >= num_sms) return 1;
  // Enough ranges to fill every SM once, each range at least 4 key blocks long.
  long long want = (num_sms + units - 1) / units;
  const long long most = nkv / 4 > 1 ? nkv / 4 : 1;
  if (want > most) want = most;
  if (want > 256) want = 256;
  return effective_splits(nkv, (int)want);
}

int fa_fwd_split(const void* q, const void* k, const void* v, const float* mask, void* out,
                 float* lse, int B, int H, int Nq, int Nk, int D, float scale, int num_splits,
                 void* workspace, size_t workspace_bytes, void* stream) {
  if (num_splits < 1) return FA_ERR_INVALID_ARGUMENT;
  Shape sh;
  int rc = validate(q, k, v, mask, out, lse, B, H, Nq, Nk, D, scale, &sh);
  if (rc != FA_OK) return rc;
  const int splits = effective_splits((Nk + 127) / 128, num_splits);
  if (splits > 1) {
    if (!workspace || !aligned16(workspace)) return FA_ERR_INVALID_ARGUMENT;
    if (workspace_bytes < fa_split_workspace_bytes(B, H, Nq, D, splits)) return FA_ERR_INVALID_ARGUMENT;
    if (workspace_overlaps(workspace, workspace_bytes, q, k, v, mask, out, lse, sh))
      return FA_ERR_INVALID_ARGUMENT;
    // Split units: checked in 64 bits before the int32 product is formed.
    if (sh.BH * sh.upb * splits > INT_MAX) return FA_ERR_INVALID_ARGUMENT;
  }
  fa::Params prm;
  DeviceState* st = nullptr;
  rc = setup(q, k, v, mask, out, lse, H, Nq, Nk, D, scale, sh, &prm, &st);
  if (rc != FA_OK) return rc;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (splits == 1) return launch_fwd(prm, *st, D, s);

  const size_t rows = (size_t)prm.BH * Nq;
  const size_t o_bytes = align256(rows * splits * D * sizeof(float));
  prm.num_splits = splits;
  prm.div_splits = fa::FastDiv::make((uint32_t)splits);
  prm.num_units = (int)(sh.BH * sh.upb * splits);
  prm.part_o = reinterpret_cast<float*>(workspace);
  prm.part_lse = reinterpret_cast<float*>(reinterpret_cast<char*>(workspace) + o_bytes);
  rc = launch_fwd(prm, *st, D, s);
  if (rc != FA_OK) return rc;
  return launch_merge(prm.part_o, prm.part_lse, prm.out, lse, splits, (long long)rows, D, s);
}

// ---------------------------------------------------------------------------
// fa_fwd_split_noalloc: the split-key forward for callers that must not
// allocate device memory — for example a plugin inside a host application
// that owns every device allocation, or a latency-critical path where
// cudaMalloc (which can synchronise the device) is not acceptable.  Its
// scratch is a fixed array inside this library.  A __device__ array's name in
// host code is only a host-side stand-in, so its device address is looked up
// with cudaGetSymbolAddress, once per device, with that device current; that
// look-up happens on the first call on each device that uses more than one
// key range.
// ---------------------------------------------------------------------------
int fa_fwd_split_noalloc(const void* q, const void* k, const void* v, const float* mask, void* out,
                         float* lse, int B, int H, int Nq, int Nk, int D, float scale,
                         int num_splits, void* stream) {
  // ---- validation: no CUDA call before this block passes ----
  if (num_splits < 1) return FA_ERR_INVALID_ARGUMENT;
  Shape sh;
  const int rc = validate(q, k, v, mask, out, lse, B, H, Nq, Nk, D, scale, &sh);
  if (rc != FA_OK) return rc;
  const int splits = effective_splits((Nk + 127) / 128, num_splits);
  if (splits > 1 && fa_split_workspace_bytes(B, H, Nq, D, splits) > (size_t)FA_NOALLOC_SCRATCH_BYTES)
    return FA_ERR_INVALID_ARGUMENT;  // does not fit the fixed scratch
  // One key range needs no scratch: fa_fwd_split then launches the plain forward.
  void* scratch = nullptr;
  if (splits > 1) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return FA_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_mutex);
    if (!g_noalloc_scratch_addr[dev]) {
      void* addr = nullptr;
      if (cudaGetSymbolAddress(&addr, g_noalloc_scratch) != cudaSuccess || addr == nullptr)
        return FA_ERR_CUDA;
      g_noalloc_scratch_addr[dev] = addr;
    }
    scratch = g_noalloc_scratch_addr[dev];
  }
  // Every partial result the merge reads is written first by the forward, so
  // nothing in the scratch needs clearing between calls.
  return fa_fwd_split(q, k, v, mask, out, lse, B, H, Nq, Nk, D, scale, splits, scratch,
                      scratch ? (size_t)FA_NOALLOC_SCRATCH_BYTES : 0, stream);
}

size_t fa_window_workspace_bytes(int B, int H, int img_h, int img_w, int D) {
  (void)B;
  (void)H;
  (void)img_h;
  (void)img_w;
  (void)D;
  return 0;  // the attention kernel gathers and scatters the window rows itself
}

int fa_fwd_window(const void* q, const void* k, const void* v, void* out, float* lse, int B, int H,
                  int img_h, int img_w, int D, int win_h, int win_w, int shift_h, int shift_w,
                  float scale, void* workspace, size_t workspace_bytes, void* stream) {
  (void)workspace;  // no scratch is used (see fa.h)
  (void)workspace_bytes;
  // ---- validation: no CUDA call before this block passes ----
  if (!q || !k || !v || !out || !lse) return FA_ERR_INVALID_ARGUMENT;
  if (B < 1 || H < 1 || img_h < 1 || img_w < 1 || win_h < 1 || win_w < 1)
    return FA_ERR_INVALID_ARGUMENT;
  if (img_h % win_h || img_w % win_w) return FA_ERR_INVALID_ARGUMENT;
  if (D != 32 && D != 64 && D != 128) return FA_ERR_UNSUPPORTED;
  if (!std::isfinite(scale)) return FA_ERR_INVALID_ARGUMENT;
  if ((int64_t)img_h * img_w > INT_MAX) return FA_ERR_INVALID_ARGUMENT;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out) || !aligned16(lse))
    return FA_ERR_INVALID_ARGUMENT;
  const size_t rows = (size_t)B * H * img_h * img_w;
  // Windowed rows are indexed in 32 bits (multiply-shift division).
  if (rows >= (size_t(1) << 31)) return FA_ERR_INVALID_ARGUMENT;
  fa::WindowGeom g{B, H, img_h, img_w, win_h, win_w, 0, 0, D, 1};
  g.shift_h = ((shift_h % img_h) + img_h) % img_h;
  g.shift_w = ((shift_w % img_w) + img_w) % img_w;
  const long long nw = g.windows();
  if ((long long)B * nw > INT_MAX) return FA_ERR_INVALID_ARGUMENT;
  // Pack windows of up to 64 tokens, as many as fill two 128-row tiles, into
  // each batch entry (a divisor of the window count, so every entry is full):
  // a work unit then holds two query tiles (both softmax warpgroups busy),
  // each seeing the keys of its own windows only.
  const int Nw = g.win_tokens();
  if (Nw <= 64) {
    int pk = 256 / Nw;
    while (pk > 1 && ((long long)B * nw) % pk) --pk;
    g.pack = pk;
  }
  g.finish();
  // The batched problem over the windows, validated like fa_fwd's (its rows
  // are those of q, k, v, out and lse, in another order).
  const int entries = (int)(B * nw / g.pack), Ne = g.entry_tokens();
  Shape sh;
  int rc = validate(q, k, v, nullptr, out, lse, entries, H, Ne, Ne, D, scale, &sh);
  if (rc != FA_OK) return rc;

  // ---- set-up (CUDA calls, nothing enqueued yet) ----
  fa::Params prm;
  DeviceState* st = nullptr;
  rc = setup(q, k, v, nullptr, out, lse, H, Ne, Ne, D, scale, sh, &prm, &st);
  if (rc != FA_OK) return rc;
  prm.seg = g.pack > 1 ? Nw : 0;  // each row sees its own window only
  // Window mode: the kernel reads each windowed row of Q, K, V from its grid
  // position and writes O and LSE back there (no gather or scatter pass).
  prm.win = 1;
  prm.wg = g;
  prm.win_q = static_cast<const __nv_bfloat16*>(q);
  prm.win_k = static_cast<const __nv_bfloat16*>(k);
  prm.win_v = static_cast<const __nv_bfloat16*>(v);
  fa::log_launch("window attention: %d batch entries of %d tokens (%d windows of %dx%d each), "
                 "rows gathered and scattered by the attention kernel",
                 entries, Ne, g.pack, win_h, win_w);
  return launch_fwd(prm, *st, D, reinterpret_cast<cudaStream_t>(stream));
}

int fa_read_device_status(void* stream, int* status) {
  if (!status) return FA_ERR_INVALID_ARGUMENT;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  int value = 0;
  if (cudaMemcpyFromSymbolAsync(&value, g_device_status, sizeof(int), 0,
                                cudaMemcpyDeviceToHost, s) != cudaSuccess)
    return FA_ERR_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return FA_ERR_CUDA;
  const int zero = 0;
  if (cudaMemcpyToSymbolAsync(g_device_status, &zero, sizeof(int), 0, cudaMemcpyHostToDevice,
                              s) != cudaSuccess)
    return FA_ERR_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return FA_ERR_CUDA;
  *status = value;
  return FA_OK;
}

int fa_measure_ex2_rate(void* stream, double* ex2_per_clock_per_sm) {
  if (!ex2_per_clock_per_sm) return FA_ERR_INVALID_ARGUMENT;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return FA_ERR_CUDA;
  const int ctas = sms * fa::kDiagCtasPerSm;
  if (ctas > fa::kDiagMaxCtas) return FA_ERR_UNSUPPORTED;
  const int iters = 2048;
  long long clk[fa::kDiagMaxCtas];
  for (int rep = 0; rep < 2; ++rep)  // the first launch warms up clocks and caches
    fa::fa_ex2_rate_kernel<<<ctas, fa::kDiagThreads, 0, s>>>(iters);
  if (cudaGetLastError() != cudaSuccess) return FA_ERR_CUDA;
  if (cudaMemcpyFromSymbolAsync(clk, fa::g_diag_clk, sizeof(long long) * ctas, 0,
                                cudaMemcpyDeviceToHost, s) != cudaSuccess ||
      cudaStreamSynchronize(s) != cudaSuccess)
    return FA_ERR_CUDA;
  long long slowest = 1;
  for (int b = 0; b < ctas; ++b) slowest = clk[b] > slowest ? clk[b] : slowest;
  const double per_sm = (double)fa::kDiagCtasPerSm * fa::kDiagThreads * fa::kDiagChains * iters;
  *ex2_per_clock_per_sm = per_sm / (double)slowest;
  return FA_OK;
}

const char* fa_status_string(int status) {
  switch (status) {
    case FA_OK: return "FA_OK";
    case FA_ERR_INVALID_ARGUMENT: return "FA_ERR_INVALID_ARGUMENT";
    case FA_ERR_UNSUPPORTED: return "FA_ERR_UNSUPPORTED";
    case FA_ERR_CUDA: return "FA_ERR_CUDA";
    case FA_ERR_TIMEOUT: return "FA_ERR_TIMEOUT";
    case FA_ERR_DEBUG_CHECK: return "FA_ERR_DEBUG_CHECK";
    default: return "FA_ERR_UNKNOWN";
  }
}

int fa_debug_build(void) {
#ifdef FA_DEBUG
  return 1;
#else
  return 0;
#endif
}

int fa_debug_report(void* stream, int* record) {
  if (!record) return FA_ERR_INVALID_ARGUMENT;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  int rec[8] = {};
  if (cudaMemcpyFromSymbolAsync(rec, g_debug_record, sizeof(rec), 0, cudaMemcpyDeviceToHost, s) !=
          cudaSuccess ||
      cudaStreamSynchronize(s) != cudaSuccess)
    return FA_ERR_CUDA;
  const int zero[8] = {};
  if (cudaMemcpyToSymbolAsync(g_debug_record, zero, sizeof(zero), 0, cudaMemcpyHostToDevice, s) !=
          cudaSuccess ||
      cudaStreamSynchronize(s) != cudaSuccess)
    return FA_ERR_CUDA;
  for (int i = 0; i < 8; ++i) record[i] = rec[i];
  return FA_OK;
}

const char* fa_version(void) {
#ifdef FA_DEBUG
  return "unet_fa_fwd_gb300 0.2.0 sm_103a debug";
#else
  return "unet_fa_fwd_gb300 0.2.0 sm_103a";
#endif
}

}  // extern "C"
