// attn_api.cu -- the library's C ABI (declared in include/attn.h): argument
// checks, per-device set-up, TMA tensor-map encoding and kernel dispatch.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <atomic>
#include <cstdint>
#include <cmath>
#include <mutex>

#include "attn.h"
#include "attn_internal.cuh"

namespace attn {
namespace {

// Errors a kernel finds (a bounded wait that ran out) are recorded here, one
// word per device, and read back by attn_check().
__device__ int g_status;

constexpr int kMaxDevices = 64;
constexpr uint64_t kDefaultLimitNs = 2000000000ull;

// attn_fwd_host splits the batch into at most this many slices, so that the
// copies of one slice overlap the kernel and the copies of its neighbours.
constexpr int kHostSlices = 8;
// Copy streams per direction (slices alternate between them); two measured no
// faster than one: the host link, not the copy engines, sets the rate.
constexpr int kCopyStreams = 1;

struct DeviceInfo {
  bool ready = false;
  bool supported = false;
  int num_sms = 0;
  int* status = nullptr;
  // attn_fwd_host: copy-in and copy-out streams and the events that order
  // them with the caller's stream (created on first use; issued under
  // host_mu so that concurrent callers do not share an event in flight).
  cudaStream_t copy_in[kCopyStreams] = {}, copy_out[kCopyStreams] = {};
  cudaEvent_t ev_start = nullptr, ev_done[kCopyStreams] = {};
  cudaEvent_t ev_in[kHostSlices] = {}, ev_kernel[kHostSlices] = {};
  std::mutex host_mu;
};

std::mutex g_mu;
DeviceInfo g_dev[kMaxDevices];
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::atomic<uint64_t> g_limit_ns{kDefaultLimitNs};
std::atomic<uint64_t> g_launches{0};
std::atomic<int> g_last_cuda_error{0};

int cuda_fail(cudaError_t e) {
  g_last_cuda_error.store(static_cast<int>(e));
  return ATTN_ERR_CUDA;
}

// Per-device set-up on first use: SM count, architecture check, address of
// the status word, the driver's tensor-map encoder.
int device_info(DeviceInfo** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e);
  if (dev < 0 || dev >= kMaxDevices) return ATTN_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_mu);
  DeviceInfo& di = g_dev[dev];
  if (!di.ready) {
    int major = 0, minor = 0, sms = 0;
    if ((e = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev)) != cudaSuccess)
      return cuda_fail(e);
    if ((e = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev)) != cudaSuccess)
      return cuda_fail(e);
    if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
      return cuda_fail(e);
    di.supported = (major == 10 && minor == 3);  // the kernels are built for sm_103a only
    di.num_sms = sms;
    if (di.supported) {
      void* addr = nullptr;
      if ((e = cudaGetSymbolAddress(&addr, g_status)) != cudaSuccess) return cuda_fail(e);
      di.status = static_cast<int*>(addr);
    }
    if (g_encode == nullptr) {
      void* fn = nullptr;
      cudaDriverEntryPointQueryResult q;
      e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                           &q);
      if (e != cudaSuccess) return cuda_fail(e);
      if (q != cudaDriverEntryPointSuccess || fn == nullptr) return cuda_fail(cudaErrorNotSupported);
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    }
    di.ready = true;
  }
  if (!di.supported) return ATTN_ERR_UNSUPPORTED;
  *out = &di;
  return ATTN_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int check_common(const void* q, const void* k, const void* v, const void* o, const float* lse,
                 int B, int h, int n_q, int n_k, int d_k, float scale, int mask_kind,
                 const int* key_lens, size_t elem) {
  if (!q || !k || !v || !o) return ATTN_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o)) return ATTN_ERR_INVALID_ARG;
  if (lse && (reinterpret_cast<uintptr_t>(lse) & 3u)) return ATTN_ERR_INVALID_ARG;
  if (B < 1 || h < 1 || n_q < 1 || n_k < 1 || d_k < 1) return ATTN_ERR_INVALID_ARG;
  if (!(std::isfinite(scale) && scale > 0.f)) return ATTN_ERR_INVALID_ARG;
  if (mask_kind != ATTN_MASK_NONE && mask_kind != ATTN_MASK_CAUSAL &&
      mask_kind != ATTN_MASK_KEY_PADDING)
    return ATTN_ERR_INVALID_ARG;
  if (mask_kind == ATTN_MASK_KEY_PADDING &&
      (key_lens == nullptr || (reinterpret_cast<uintptr_t>(key_lens) & 3u)))
    return ATTN_ERR_INVALID_ARG;
  // Index arithmetic: B*h fits a TMA coordinate and a grid; every tensor
  // stays below 2^40 bytes (the TMA stride limit).
  const long long bh = static_cast<long long>(B) * h;
  if (bh > 0x7fffffffLL) return ATTN_ERR_INVALID_ARG;
  const long long n = n_q > n_k ? n_q : n_k;
  if (bh * n * d_k * static_cast<long long>(elem) >= (1LL << 40)) return ATTN_ERR_INVALID_ARG;
  return ATTN_OK;
}

// (d, n, B*H) fp32 view with a (min(d, 32), 64, 1) box in the swizzle of its
// 4*min(d, 32)-byte rows (the backward's dQ accumulator, added into by TMA
// reduce).
int encode_3d_f32(CUtensorMap* map, const void* base, int d, int n, long long bh) {
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(n),
                        static_cast<cuuint64_t>(bh)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(d) * 4,
                           static_cast<cuuint64_t>(d) * 4 * static_cast<cuuint64_t>(n)};
  const int inner = d < 32 ? d : 32;
  cuuint32_t box[3] = {static_cast<cuuint32_t>(inner), 64u, 1u};
  cuuint32_t estr[3] = {1u, 1u, 1u};
  const CUtensorMapSwizzle swz = inner == 32   ? CU_TENSOR_MAP_SWIZZLE_128B
                                 : inner == 16 ? CU_TENSOR_MAP_SWIZZLE_64B
                                               : CU_TENSOR_MAP_SWIZZLE_32B;
  CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<void*>(base), dims,
                        strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swz,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? ATTN_OK : cuda_fail(cudaErrorInvalidValue);
}

// Head sizes the tensor-core forward covers.
bool tc_head_size(int d) { return d == 16 || d == 32 || d == 64 || d == 128; }

// Element strides of a [B, h, n, d] tensor view (d contiguous).
using Strides = RowStrides;

Strides bhsd(int h, int n, int d) {
  return Strides{static_cast<long long>(h) * n * d, static_cast<long long>(n) * d, d};
}

// A stride the TMA can use: positive and a multiple of 16 bytes.
bool stride_ok(long long elems) {
  return elems > 0 && (elems * 2) % 16 == 0 && elems * 2 < (1LL << 40);
}

// (d, n, h, B) bf16 view with the given strides and a (min(d, 64), rows, 1, 1)
// box in the widest swizzle its 2*min(d, 64)-byte rows fit.
int encode_4d(CUtensorMap* map, const void* base, int d, int n, int h, int B, Strides st,
              int box_rows) {
  cuuint64_t dims[4] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(n),
                        static_cast<cuuint64_t>(h), static_cast<cuuint64_t>(B)};
  cuuint64_t strides[3] = {static_cast<cuuint64_t>(st.n) * 2, static_cast<cuuint64_t>(st.h) * 2,
                           static_cast<cuuint64_t>(st.b) * 2};
  const int inner = d < 64 ? d : 64;
  const CUtensorMapSwizzle swz = inner == 64   ? CU_TENSOR_MAP_SWIZZLE_128B
                                 : inner == 32 ? CU_TENSOR_MAP_SWIZZLE_64B
                                               : CU_TENSOR_MAP_SWIZZLE_32B;
  cuuint32_t box[4] = {static_cast<cuuint32_t>(inner), static_cast<cuuint32_t>(box_rows), 1u, 1u};
  cuuint32_t estr[4] = {1u, 1u, 1u, 1u};
  CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), dims,
                        strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swz,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? ATTN_OK : ATTN_ERR_INVALID_ARG;
}

// The forward's four maps: Q and O with 128-row boxes, K and V with the key
// tile of this head size.  st = strides of q, k, v, o, or null for
// contiguous [B, h, n, d].
int encode_fwd_maps(CUtensorMap* tmq, CUtensorMap* tmk, CUtensorMap* tmv, CUtensorMap* tmo,
                    const void* q, const void* k, const void* v, const void* o, int d, int n_q,
                    int n_k, int h, int B, const Strides* st) {
  const int kv_rows = fwd_tc_kv_rows(d);
  const Strides sq = st ? st[0] : bhsd(h, n_q, d), sk = st ? st[1] : bhsd(h, n_k, d),
                sv = st ? st[2] : bhsd(h, n_k, d), so = st ? st[3] : bhsd(h, n_q, d);
  int rc;
  if ((rc = encode_4d(tmq, q, d, n_q, h, B, sq, 128)) != ATTN_OK) return rc;
  if ((rc = encode_4d(tmk, k, d, n_k, h, B, sk, kv_rows)) != ATTN_OK) return rc;
  if ((rc = encode_4d(tmv, v, d, n_k, h, B, sv, kv_rows)) != ATTN_OK) return rc;
  return encode_4d(tmo, o, d, n_q, h, B, so, 128);
}

int encode_2d(CUtensorMap* map, const void* base) {
  cuuint64_t dims[2] = {64, 128};
  cuuint64_t strides[1] = {128};
  cuuint32_t box[2] = {64, 128};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims,
                        strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? ATTN_OK : cuda_fail(cudaErrorInvalidValue);
}

// Scratch for attn_decode_noalloc: a fixed-size array in the library's own
// device memory, created when the library's module is loaded on a device and
// kept until the process exits.  Host code only knows the symbol; the device
// address is looked up once per device (scratch_on_device) and handed to the
// kernels as a plain pointer.
static __device__ __align__(256) unsigned char g_decode_scratch[ATTN_DECODE_NOALLOC_SCRATCH_BYTES];
void* g_scratch_addr[kMaxDevices] = {};

// Device address of g_decode_scratch on the current device (looked up on the
// first call per device, under the set-up lock).
int scratch_on_device(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e);
  if (dev < 0 || dev >= kMaxDevices) return ATTN_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_mu);
  if (g_scratch_addr[dev] == nullptr) {
    void* addr = nullptr;
    if ((e = cudaGetSymbolAddress(&addr, g_decode_scratch)) != cudaSuccess) return cuda_fail(e);
    if (addr == nullptr) return cuda_fail(cudaErrorInvalidSymbol);
    g_scratch_addr[dev] = addr;
  }
  *out = g_scratch_addr[dev];
  return ATTN_OK;
}

// K and V caches with 128-key boxes, then with 32-key boxes for partial tiles.
int encode_decode_maps(CUtensorMap* maps, const void* k_cache, const void* v_cache, int d_k,
                       int L_max, int B, int h, Strides sk, Strides sv) {
  int rc;
  if ((rc = encode_4d(&maps[0], k_cache, d_k, L_max, h, B, sk, 128)) != ATTN_OK) return rc;
  if ((rc = encode_4d(&maps[1], v_cache, d_k, L_max, h, B, sv, 128)) != ATTN_OK) return rc;
  if ((rc = encode_4d(&maps[2], k_cache, d_k, L_max, h, B, sk, 32)) != ATTN_OK) return rc;
  return encode_4d(&maps[3], v_cache, d_k, L_max, h, B, sv, 32);
}

// Device staging of attn_fwd_host: Q, K, V, O (bf16), LSE (fp32) and the key
// lengths (int32), each at a 256-byte boundary, for the whole batch.
struct HostLayout {
  size_t q, k, v, o, lse, lens, bytes;
};

HostLayout host_layout(int B, int h, int n_q, int n_k, int d) {
  auto up = [](size_t x) { return (x + 255) & ~static_cast<size_t>(255); };
  const size_t bh = static_cast<size_t>(B) * h;
  HostLayout l;
  size_t off = 0;
  l.q = off;
  off += up(bh * n_q * d * 2);
  l.k = off;
  off += up(bh * n_k * d * 2);
  l.v = off;
  off += up(bh * n_k * d * 2);
  l.o = off;
  off += up(bh * n_q * d * 2);
  l.lse = off;
  off += up(bh * n_q * 4);
  l.lens = off;
  off += up(static_cast<size_t>(B) * 4);
  l.bytes = off;
  return l;
}

// The copy streams and events of attn_fwd_host, created once per device.
int host_streams(DeviceInfo* di) {
  std::lock_guard<std::mutex> lock(g_mu);
  if (di->copy_in[0] != nullptr) return ATTN_OK;
  cudaError_t e;
  cudaStream_t st[2 * kCopyStreams];
  for (int i = 0; i < 2 * kCopyStreams; ++i)
    if ((e = cudaStreamCreateWithFlags(&st[i], cudaStreamNonBlocking)) != cudaSuccess)
      return cuda_fail(e);
  cudaEvent_t* evs[1 + kCopyStreams + 2 * kHostSlices];
  int n = 0;
  evs[n++] = &di->ev_start;
  for (int i = 0; i < kCopyStreams; ++i) evs[n++] = &di->ev_done[i];
  for (int i = 0; i < kHostSlices; ++i) {
    evs[n++] = &di->ev_in[i];
    evs[n++] = &di->ev_kernel[i];
  }
  for (int i = 0; i < n; ++i)
    if ((e = cudaEventCreateWithFlags(evs[i], cudaEventDisableTiming)) != cudaSuccess)
      return cuda_fail(e);
  for (int i = kCopyStreams - 1; i >= 0; --i) {
    di->copy_out[i] = st[kCopyStreams + i];
    di->copy_in[i] = st[i];  // copy_in[0] last: marks the set as complete
  }
  return ATTN_OK;
}

LaunchCtx make_ctx(const DeviceInfo& di, cudaStream_t stream) {
  LaunchCtx ctx;
  ctx.num_sms = di.num_sms;
  ctx.limit_ns = g_limit_ns.load();
  ctx.status = di.status;
  ctx.stream = stream;
  return ctx;
}

}  // namespace
}  // namespace attn

using namespace attn;

extern "C" {

int attn_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int h,
             int n_q, int n_k, int d_k, float scale, int mask_kind, const int* key_lens,
             struct CUstream_st* stream) {
  int rc = check_common(q, k, v, o, lse, B, h, n_q, n_k, d_k, scale, mask_kind, key_lens, 2);
  if (rc != ATTN_OK) return rc;
  if (!tc_head_size(d_k)) return ATTN_ERR_UNSUPPORTED;
  DeviceInfo* di = nullptr;
  if ((rc = device_info(&di)) != ATTN_OK) return rc;
  CUtensorMap tmq, tmk, tmv, tmo;
  if ((rc = encode_fwd_maps(&tmq, &tmk, &tmv, &tmo, q, k, v, o, d_k, n_q, n_k, h, B, nullptr)) !=
      ATTN_OK)
    return rc;
  Problem pb{q, k, v, o, lse, B, h, n_q, n_k, d_k, scale, mask_kind,
             mask_kind == ATTN_MASK_KEY_PADDING ? key_lens : nullptr};
  cudaError_t e = launch_fwd_tc(pb, tmq, tmk, tmv, tmo, make_ctx(*di, stream));
  if (e != cudaSuccess) return cuda_fail(e);
  g_launches.fetch_add(1);
  return ATTN_OK;
}

int attn_fwd_window(const void* q, const void* k, const void* v, void* o, float* lse, int B, int h,
                    int n_q, int n_k, int d_k, float scale, int window_left, int window_right,
                    struct CUstream_st* stream) {
  int rc = check_common(q, k, v, o, lse, B, h, n_q, n_k, d_k, scale, ATTN_MASK_NONE, nullptr, 2);
  if (rc != ATTN_OK) return rc;
  if (window_left < 0 || window_right < 0) return ATTN_ERR_INVALID_ARG;
  if (!tc_head_size(d_k)) return ATTN_ERR_UNSUPPORTED;
  DeviceInfo* di = nullptr;
  if ((rc = device_info(&di)) != ATTN_OK) return rc;
  CUtensorMap tmq, tmk, tmv, tmo;
  if ((rc = encode_fwd_maps(&tmq, &tmk, &tmv, &tmo, q, k, v, o, d_k, n_q, n_k, h, B, nullptr)) !=
      ATTN_OK)
    return rc;
  // a side longer than both sequences changes nothing; clamping keeps the
  // kernel's index arithmetic within int
  const int reach = n_q + n_k;
  Problem pb{q, k, v, o, lse, B, h, n_q, n_k, d_k, scale, kMaskBand, nullptr,
             window_left < reach ? window_left : reach, window_right < reach ? window_right : reach};
  cudaError_t e = launch_fwd_tc(pb, tmq, tmk, tmv, tmo, make_ctx(*di, stream));
  if (e != cudaSuccess) return cuda_fail(e);
  g_launches.fetch_add(1);
  return ATTN_OK;
}

int attn_fwd_strided(const void* q, const void* k, const void* v, void* o, float* lse, int B,
                     int h, int n_q, int n_k, int d_k, const int64_t* q_strides,
                     const int64_t* k_strides, const int64_t* v_strides, const int64_t* o_strides,
                     float scale, int mask_kind, const int* key_lens, int window_left,
                     int window_right, struct CUstream_st* stream) {
  if (!q || !k || !v || !o) return ATTN_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o)) return ATTN_ERR_INVALID_ARG;
  if (lse && (reinterpret_cast<uintptr_t>(lse) & 3u)) return ATTN_ERR_INVALID_ARG;
  if (B < 1 || h < 1 || n_q < 1 || n_k < 1 || d_k < 1) return ATTN_ERR_INVALID_ARG;
  if (!(std::isfinite(scale) && scale > 0.f)) return ATTN_ERR_INVALID_ARG;
  if (mask_kind < ATTN_MASK_NONE || mask_kind > ATTN_MASK_WINDOW) return ATTN_ERR_INVALID_ARG;
  if (mask_kind == ATTN_MASK_KEY_PADDING &&
      (key_lens == nullptr || (reinterpret_cast<uintptr_t>(key_lens) & 3u)))
    return ATTN_ERR_INVALID_ARG;
  if (mask_kind == ATTN_MASK_WINDOW && (window_left < 0 || window_right < 0))
    return ATTN_ERR_INVALID_ARG;
  if (!q_strides || !k_strides || !v_strides || !o_strides) return ATTN_ERR_INVALID_ARG;
  if (static_cast<long long>(B) * h > 0x7fffffffLL) return ATTN_ERR_INVALID_ARG;
  Strides st[4];
  const int64_t* in[4] = {q_strides, k_strides, v_strides, o_strides};
  for (int i = 0; i < 4; ++i) {
    st[i] = Strides{in[i][0], in[i][1], in[i][2]};
    if (!stride_ok(st[i].b) || !stride_ok(st[i].h) || !stride_ok(st[i].n))
      return ATTN_ERR_INVALID_ARG;
  }
  if (!tc_head_size(d_k)) return ATTN_ERR_UNSUPPORTED;
  DeviceInfo* di = nullptr;
  int rc;
  if ((rc = device_info(&di)) != ATTN_OK) return rc;
  CUtensorMap tmq, tmk, tmv, tmo;
  if ((rc = encode_fwd_maps(&tmq, &tmk, &tmv, &tmo, q, k, v, o, d_k, n_q, n_k, h, B, st)) !=
      ATTN_OK)
    return rc;
  const int reach = n_q + n_k;
  Problem pb{q, k, v, o, lse, B, h, n_q, n_k, d_k, scale,
             mask_kind == ATTN_MASK_WINDOW ? static_cast<int>(kMaskBand) : mask_kind,
             mask_kind == ATTN_MASK_KEY_PADDING ? key_lens : nullptr,
             window_left < reach ? window_left : reach, window_right < reach ? window_right : reach};
  cudaError_t e = launch_fwd_tc(pb, tmq, tmk, tmv, tmo, make_ctx(*di, stream));
  if (e != cudaSuccess) return cuda_fail(e);
  g_launches.fetch_add(1);
  return ATTN_OK;
}

size_t attn_fwd_host_buffer_bytes(int B, int h, int n_q, int n_k, int d_k) {
  if (B < 1 || h < 1 || n_q < 1 || n_k < 1 || !tc_head_size(d_k)) return 0;
  if (static_cast<long long>(B) * h > 0x7fffffffLL) return 0;
  return host_layout(B, h, n_q, n_k, d_k).bytes;
}

int attn_fwd_host(const void* q, const void* k, const void* v, void* o, float* lse, int B, int h,
                  int n_q, int n_k, int d_k, float scale, int mask_kind, const int* key_lens,
                  int window_left, int window_right, void* dev_buf, size_t dev_buf_bytes,
                  struct CUstream_st* stream) {
  const bool window = mask_kind == ATTN_MASK_WINDOW;
  if (mask_kind < ATTN_MASK_NONE || mask_kind > ATTN_MASK_WINDOW) return ATTN_ERR_INVALID_ARG;
  if (window && (window_left < 0 || window_right < 0)) return ATTN_ERR_INVALID_ARG;
  if (!q || !k || !v || !o) return ATTN_ERR_INVALID_ARG;
  if (mask_kind == ATTN_MASK_KEY_PADDING && key_lens == nullptr) return ATTN_ERR_INVALID_ARG;
  // sizes, scale and the device-side limits, checked as for attn_fwd on the
  // staging buffer (the host buffers need no alignment)
  const void* stage = dev_buf;
  int rc = check_common(stage, stage, stage, stage, nullptr, B, h, n_q, n_k, d_k, scale,
                        mask_kind == ATTN_MASK_KEY_PADDING ? ATTN_MASK_KEY_PADDING : ATTN_MASK_NONE,
                        static_cast<const int*>(stage), 2);
  if (rc != ATTN_OK) return rc;
  if (reinterpret_cast<uintptr_t>(dev_buf) & 255u) return ATTN_ERR_INVALID_ARG;
  if (!tc_head_size(d_k)) return ATTN_ERR_UNSUPPORTED;
  const HostLayout lay = host_layout(B, h, n_q, n_k, d_k);
  if (dev_buf_bytes < lay.bytes) return ATTN_ERR_INVALID_ARG;
  DeviceInfo* di = nullptr;
  if ((rc = device_info(&di)) != ATTN_OK) return rc;
  if ((rc = host_streams(di)) != ATTN_OK) return rc;
  std::lock_guard<std::mutex> lock(di->host_mu);

  uint8_t* dbuf = static_cast<uint8_t*>(dev_buf);
  const size_t qrow = static_cast<size_t>(h) * n_q * d_k * 2;  // bytes of one batch entry
  const size_t krow = static_cast<size_t>(h) * n_k * d_k * 2;
  const size_t lrow = static_cast<size_t>(h) * n_q * 4;
  const bool padding = mask_kind == ATTN_MASK_KEY_PADDING;
  const int reach = n_q + n_k;
  const int slices = B < kHostSlices ? B : kHostSlices;
  cudaError_t e;
  // the staging buffer and the host buffers may still be in use by work
  // enqueued earlier on the caller's stream
  if ((e = cudaEventRecord(di->ev_start, stream)) != cudaSuccess) return cuda_fail(e);
  for (int i = 0; i < kCopyStreams; ++i) {
    if ((e = cudaStreamWaitEvent(di->copy_in[i], di->ev_start, 0)) != cudaSuccess)
      return cuda_fail(e);
    if ((e = cudaStreamWaitEvent(di->copy_out[i], di->ev_start, 0)) != cudaSuccess)
      return cuda_fail(e);
  }
  const cudaMemcpyKind h2d = cudaMemcpyHostToDevice, d2h = cudaMemcpyDeviceToHost;
  for (int s = 0; s < slices; ++s) {
    const int b0 = static_cast<int>(static_cast<long long>(B) * s / slices);
    const int b1 = static_cast<int>(static_cast<long long>(B) * (s + 1) / slices);
    const int nb = b1 - b0;
    uint8_t* dq = dbuf + lay.q + b0 * qrow;
    uint8_t* dk = dbuf + lay.k + b0 * krow;
    uint8_t* dv = dbuf + lay.v + b0 * krow;
    uint8_t* dout = dbuf + lay.o + b0 * qrow;
    float* dlse = reinterpret_cast<float*>(dbuf + lay.lse + b0 * lrow);
    int* dlens = reinterpret_cast<int*>(dbuf + lay.lens) + b0;
    cudaStream_t copy_in = di->copy_in[s % kCopyStreams];
    cudaStream_t copy_out = di->copy_out[s % kCopyStreams];
    // copy in (one copy per tensor slice)
    if ((e = cudaMemcpyAsync(dq, static_cast<const uint8_t*>(q) + b0 * qrow, nb * qrow, h2d,
                             copy_in)) != cudaSuccess)
      return cuda_fail(e);
    if ((e = cudaMemcpyAsync(dk, static_cast<const uint8_t*>(k) + b0 * krow, nb * krow, h2d,
                             copy_in)) != cudaSuccess)
      return cuda_fail(e);
    if ((e = cudaMemcpyAsync(dv, static_cast<const uint8_t*>(v) + b0 * krow, nb * krow, h2d,
                             copy_in)) != cudaSuccess)
      return cuda_fail(e);
    if (padding && (e = cudaMemcpyAsync(dlens, key_lens + b0, nb * sizeof(int), h2d, copy_in)) !=
                       cudaSuccess)
      return cuda_fail(e);
    if ((e = cudaEventRecord(di->ev_in[s], copy_in)) != cudaSuccess) return cuda_fail(e);
    // the forward of this slice on the caller's stream
    if ((e = cudaStreamWaitEvent(stream, di->ev_in[s], 0)) != cudaSuccess) return cuda_fail(e);
    CUtensorMap tmq, tmk, tmv, tmo;
    if ((rc = encode_fwd_maps(&tmq, &tmk, &tmv, &tmo, dq, dk, dv, dout, d_k, n_q, n_k, h, nb,
                              nullptr)) != ATTN_OK)
      return rc;
    Problem pb{dq, dk, dv, dout, lse ? dlse : nullptr, nb, h, n_q, n_k, d_k, scale,
               window ? static_cast<int>(kMaskBand) : mask_kind, padding ? dlens : nullptr,
               window_left < reach ? window_left : reach,
               window_right < reach ? window_right : reach};
    if ((e = launch_fwd_tc(pb, tmq, tmk, tmv, tmo, make_ctx(*di, stream))) != cudaSuccess)
      return cuda_fail(e);
    g_launches.fetch_add(1);
    if ((e = cudaEventRecord(di->ev_kernel[s], stream)) != cudaSuccess) return cuda_fail(e);
    // copy out
    if ((e = cudaStreamWaitEvent(copy_out, di->ev_kernel[s], 0)) != cudaSuccess) return cuda_fail(e);
    if ((e = cudaMemcpyAsync(static_cast<uint8_t*>(o) + b0 * qrow, dout, nb * qrow, d2h,
                             copy_out)) != cudaSuccess)
      return cuda_fail(e);
    if (lse && (e = cudaMemcpyAsync(reinterpret_cast<uint8_t*>(lse) + b0 * lrow, dlse, nb * lrow,
                                    d2h, copy_out)) != cudaSuccess)
      return cuda_fail(e);
  }
  // the caller's stream resumes once every copy out is done
  for (int i = 0; i < kCopyStreams; ++i) {
    if ((e = cudaEventRecord(di->ev_done[i], di->copy_out[i])) != cudaSuccess) return cuda_fail(e);
    if ((e = cudaStreamWaitEvent(stream, di->ev_done[i], 0)) != cudaSuccess) return cuda_fail(e);
  }
  return ATTN_OK;
}

int attn_fwd_f32(const float* q, const float* k, const float* v, float* o, float* lse, int B,
                 int h, int n_q, int n_k, int d_k, float scale, int mask_kind,
                 const int* key_lens, struct CUstream_st* stream) {
  int rc = check_common(q, k, v, o, lse, B, h, n_q, n_k, d_k, scale, mask_kind, key_lens, 4);
  if (rc != ATTN_OK) return rc;
  if (d_k != 16 && d_k != 32 && d_k != 64 && d_k != 128) return ATTN_ERR_UNSUPPORTED;
  if (static_cast<long long>(B) * h > 65535) return ATTN_ERR_UNSUPPORTED;  // grid.y
  DeviceInfo* di = nullptr;
  if ((rc = device_info(&di)) != ATTN_OK) return rc;
  Problem pb{q, k, v, o, lse, B, h, n_q, n_k, d_k, scale, mask_kind,
             mask_kind == ATTN_MASK_KEY_PADDING ? key_lens : nullptr};
  cudaError_t e = launch_fwd_f32(pb, make_ctx(*di, stream));
  if (e != cudaSuccess) return cuda_fail(e);
  g_launches.fetch_add(1);
  return ATTN_OK;
}

size_t attn_decode_workspace_bytes(int B, int h, int n_q, int L_max, int d_k) {
  if (B < 1 || h < 1 || n_q < 1 || n_q > kDecodeMaxQueries || L_max < 1 || !tc_head_size(d_k))
    return 0;
  DeviceInfo* di = nullptr;
  if (device_info(&di) != ATTN_OK) return 0;
  return decode_plan(B, h, n_q, L_max, d_k, di->num_sms).workspace_bytes;
}

size_t attn_decode_window_workspace_bytes(int B, int h, int n_q, int L_max, int d_k, int window) {
  if (window < 0) return 0;
  // the splits cover the window's keys only
  return attn_decode_workspace_bytes(B, h, n_q, window < L_max ? window + 1 : L_max, d_k);
}

}  // extern "C"

namespace attn {
namespace {
// st: strides of q, k_cache, v_cache, o, or null for contiguous tensors.
// scratch_noalloc: take the partials' space from the library's own array
// instead of the caller's workspace.  window: restricted self-attention
// (keys [len - 1 - window, len)), or -1 for all cached keys.
static int decode_impl(const void* q, const void* k_cache, const void* v_cache, void* o,
                       float* lse, int B, int h, int n_q, int L_max, int d_k, const Strides* st,
                       float scale, const int* cache_lens, void* workspace,
                       size_t workspace_bytes, bool scratch_noalloc, struct CUstream_st* stream,
                       int window = -1) {
  int rc = check_common(q, k_cache, v_cache, o, lse, B, h, n_q, L_max, d_k, scale,
                        ATTN_MASK_NONE, nullptr, 2);
  if (rc != ATTN_OK) return rc;
  if (cache_lens && (reinterpret_cast<uintptr_t>(cache_lens) & 3u)) return ATTN_ERR_INVALID_ARG;
  if (!tc_head_size(d_k) || n_q > kDecodeMaxQueries) return ATTN_ERR_UNSUPPORTED;
  if (static_cast<long long>(B) * h > 65535) return ATTN_ERR_UNSUPPORTED;  // grid.y
  DeviceInfo* di = nullptr;
  if ((rc = device_info(&di)) != ATTN_OK) return rc;
  // the most keys one query sees: what the cache is split by
  const int seen = window >= 0 && window < L_max ? window + 1 : L_max;
  const DecodePlan plan = decode_plan(B, h, n_q, seen, d_k, di->num_sms);
  if (scratch_noalloc) {
    if (plan.workspace_bytes > ATTN_DECODE_NOALLOC_SCRATCH_BYTES)
      return ATTN_ERR_SCRATCH_TOO_SMALL;
    // only a split cache writes partials: the array is not touched otherwise
    workspace = nullptr;
    if (plan.workspace_bytes > 0 && (rc = scratch_on_device(&workspace)) != ATTN_OK) return rc;
  } else if (plan.workspace_bytes > 0 && (workspace == nullptr ||
                                          workspace_bytes < plan.workspace_bytes ||
                                          !aligned16(workspace))) {
    return ATTN_ERR_INVALID_ARG;
  }
  const Strides sq = st ? st[0] : bhsd(h, n_q, d_k), sk = st ? st[1] : bhsd(h, L_max, d_k),
                sv = st ? st[2] : bhsd(h, L_max, d_k), so = st ? st[3] : bhsd(h, n_q, d_k);
  CUtensorMap maps[4];
  if (d_k == 64 &&
      (rc = encode_decode_maps(maps, k_cache, v_cache, d_k, L_max, B, h, sk, sv)) != ATTN_OK)
    return rc;
  DecodeProblem pb{q,  k_cache, v_cache, o,          lse, B,  h,  n_q, L_max,
                   d_k, scale,  cache_lens, sq, sk, sv, so, window};
  cudaError_t e = launch_decode(pb, maps, plan, static_cast<float*>(workspace),
                                make_ctx(*di, stream));
  if (e != cudaSuccess) return cuda_fail(e);
  g_launches.fetch_add(plan.splits > 1 ? 2 : 1);
  return ATTN_OK;
}
}  // namespace
}  // namespace attn

extern "C" {

int attn_decode(const void* q, const void* k_cache, const void* v_cache, void* o, float* lse,
                int B, int h, int n_q, int L_max, int d_k, float scale, const int* cache_lens,
                void* workspace, size_t workspace_bytes, struct CUstream_st* stream) {
  return decode_impl(q, k_cache, v_cache, o, lse, B, h, n_q, L_max, d_k, nullptr, scale,
                     cache_lens, workspace, workspace_bytes, false, stream);
}

int attn_decode_window(const void* q, const void* k_cache, const void* v_cache, void* o,
                       float* lse, int B, int h, int n_q, int L_max, int d_k, float scale,
                       const int* cache_lens, int window, void* workspace,
                       size_t workspace_bytes, struct CUstream_st* stream) {
  if (window < 0) return ATTN_ERR_INVALID_ARG;
  return decode_impl(q, k_cache, v_cache, o, lse, B, h, n_q, L_max, d_k, nullptr, scale,
                     cache_lens, workspace, workspace_bytes, false, stream, window);
}

int attn_decode_noalloc(const void* q, const void* k_cache, const void* v_cache, void* o,
                        float* lse, int B, int h, int n_q, int L_max, int d_k, float scale,
                        const int* cache_lens, struct CUstream_st* stream) {
  return decode_impl(q, k_cache, v_cache, o, lse, B, h, n_q, L_max, d_k, nullptr, scale,
                     cache_lens, nullptr, 0, true, stream);
}

int attn_decode_strided(const void* q, const void* k_cache, const void* v_cache, void* o,
                        float* lse, int B, int h, int n_q, int L_max, int d_k,
                        const int64_t* strides, float scale, const int* cache_lens,
                        void* workspace, size_t workspace_bytes, struct CUstream_st* stream) {
  if (strides == nullptr) return ATTN_ERR_INVALID_ARG;
  Strides st[4];
  for (int i = 0; i < 4; ++i) {
    st[i] = Strides{strides[3 * i], strides[3 * i + 1], strides[3 * i + 2]};
    if (!stride_ok(st[i].b) || !stride_ok(st[i].h) || !stride_ok(st[i].n))
      return ATTN_ERR_INVALID_ARG;
  }
  return decode_impl(q, k_cache, v_cache, o, lse, B, h, n_q, L_max, d_k, st, scale, cache_lens,
                     workspace, workspace_bytes, false, stream);
}

size_t attn_bwd_workspace_bytes(int B, int h, int n_q, int d_k) {
  if (B < 1 || h < 1 || n_q < 1 || !bwd_head_size_ok(d_k)) return 0;
  if (static_cast<long long>(B) * h > 0x7fffffffLL) return 0;
  return bwd_layout(B, h, n_q, d_k).bytes;
}

}  // extern "C"

namespace attn {
namespace {
// st: strides of q, k, v, o, dout, dq, dk, dv, or null for contiguous
// [B, h, n, d] tensors.
static int bwd_impl(const void* q, const void* k, const void* v, const void* o, const void* dout,
                    const float* lse, void* dq, void* dk, void* dv, int B, int h, int n_q,
                    int n_k, int d_k, const Strides* st, float scale, int mask_kind,
                    const int* key_lens, int window_left, int window_right, void* workspace,
                    size_t workspace_bytes, struct CUstream_st* stream) {
  const bool window = mask_kind == kMaskBand;
  int rc = check_common(q, k, v, o, lse, B, h, n_q, n_k, d_k, scale,
                        window ? ATTN_MASK_NONE : mask_kind, key_lens, 2);
  if (rc != ATTN_OK) return rc;
  if (!dout || !lse || !dq || !dk || !dv || !workspace) return ATTN_ERR_INVALID_ARG;
  if (!aligned16(dout) || !aligned16(dq) || !aligned16(dk) || !aligned16(dv) ||
      !aligned16(workspace))
    return ATTN_ERR_INVALID_ARG;
  if (!bwd_head_size_ok(d_k)) return ATTN_ERR_UNSUPPORTED;
  const BwdLayout lay = bwd_layout(B, h, n_q, d_k);
  if (workspace_bytes < lay.bytes) return ATTN_ERR_INVALID_ARG;
  DeviceInfo* di = nullptr;
  if ((rc = device_info(&di)) != ATTN_OK) return rc;
  const long long bh = static_cast<long long>(B) * h;
  const Strides rq = bhsd(h, n_q, d_k), rk = bhsd(h, n_k, d_k);
  const Strides sq = st ? st[0] : rq, sk = st ? st[1] : rk, sv = st ? st[2] : rk,
                so = st ? st[3] : rq, sdo = st ? st[4] : rq, sdq = st ? st[5] : rq,
                sdk = st ? st[6] : rk, sdv = st ? st[7] : rk;
  CUtensorMap maps[7];
  if ((rc = encode_4d(&maps[0], q, d_k, n_q, h, B, sq, 128)) != ATTN_OK) return rc;
  if ((rc = encode_4d(&maps[1], k, d_k, n_k, h, B, sk, 128)) != ATTN_OK) return rc;
  if ((rc = encode_4d(&maps[2], v, d_k, n_k, h, B, sv, 128)) != ATTN_OK) return rc;
  if ((rc = encode_4d(&maps[3], dout, d_k, n_q, h, B, sdo, 128)) != ATTN_OK) return rc;
  if ((rc = encode_4d(&maps[4], dk, d_k, n_k, h, B, sdk, 64)) != ATTN_OK) return rc;
  if ((rc = encode_4d(&maps[5], dv, d_k, n_k, h, B, sdv, 64)) != ATTN_OK) return rc;
  if ((rc = encode_3d_f32(&maps[6], static_cast<uint8_t*>(workspace) + lay.dq_acc_off, d_k, n_q,
                          bh)) != ATTN_OK)
    return rc;
  const int reach = n_q + n_k;
  BwdProblem pb{q, k, v, o, dout, lse, dq, dk, dv, B, h, n_q, n_k, d_k, scale, mask_kind,
                mask_kind == ATTN_MASK_KEY_PADDING ? key_lens : nullptr,
                window_left < reach ? window_left : reach,
                window_right < reach ? window_right : reach, so, sdo, sdq};
  cudaError_t e = launch_bwd(pb, maps, workspace, make_ctx(*di, stream));
  if (e != cudaSuccess) return cuda_fail(e);
  g_launches.fetch_add(3);
  return ATTN_OK;
}
}  // namespace
}  // namespace attn

extern "C" {

int attn_bwd(const void* q, const void* k, const void* v, const void* o, const void* dout,
             const float* lse, void* dq, void* dk, void* dv, int B, int h, int n_q, int n_k,
             int d_k, float scale, int mask_kind, const int* key_lens, void* workspace,
             size_t workspace_bytes, struct CUstream_st* stream) {
  if (mask_kind == ATTN_MASK_WINDOW) return ATTN_ERR_INVALID_ARG;  // attn_bwd_window
  return bwd_impl(q, k, v, o, dout, lse, dq, dk, dv, B, h, n_q, n_k, d_k, nullptr, scale,
                  mask_kind, key_lens, 0, 0, workspace, workspace_bytes, stream);
}

int attn_bwd_window(const void* q, const void* k, const void* v, const void* o, const void* dout,
                    const float* lse, void* dq, void* dk, void* dv, int B, int h, int n_q,
                    int n_k, int d_k, float scale, int window_left, int window_right,
                    void* workspace, size_t workspace_bytes, struct CUstream_st* stream) {
  if (window_left < 0 || window_right < 0) return ATTN_ERR_INVALID_ARG;
  return bwd_impl(q, k, v, o, dout, lse, dq, dk, dv, B, h, n_q, n_k, d_k, nullptr, scale,
                  kMaskBand, nullptr, window_left, window_right, workspace, workspace_bytes,
                  stream);
}

int attn_bwd_strided(const void* q, const void* k, const void* v, const void* o, const void* dout,
                     const float* lse, void* dq, void* dk, void* dv, int B, int h, int n_q,
                     int n_k, int d_k, const int64_t* strides, float scale, int mask_kind,
                     const int* key_lens, int window_left, int window_right, void* workspace,
                     size_t workspace_bytes, struct CUstream_st* stream) {
  if (mask_kind < ATTN_MASK_NONE || mask_kind > ATTN_MASK_WINDOW) return ATTN_ERR_INVALID_ARG;
  if (mask_kind == ATTN_MASK_WINDOW && (window_left < 0 || window_right < 0))
    return ATTN_ERR_INVALID_ARG;
  if (strides == nullptr) return ATTN_ERR_INVALID_ARG;
  Strides st[8];
  for (int i = 0; i < 8; ++i) {
    st[i] = Strides{strides[3 * i], strides[3 * i + 1], strides[3 * i + 2]};
    if (!stride_ok(st[i].b) || !stride_ok(st[i].h) || !stride_ok(st[i].n))
      return ATTN_ERR_INVALID_ARG;
  }
  const bool window = mask_kind == ATTN_MASK_WINDOW;
  return bwd_impl(q, k, v, o, dout, lse, dq, dk, dv, B, h, n_q, n_k, d_k, st, scale,
                  window ? static_cast<int>(kMaskBand) : mask_kind, window ? nullptr : key_lens,
                  window ? window_left : 0, window ? window_right : 0, workspace,
                  workspace_bytes, stream);
}

int attn_check(struct CUstream_st* stream) {
  cudaError_t e = cudaStreamSynchronize(stream);
  if (e != cudaSuccess) return cuda_fail(e);
  DeviceInfo* di = nullptr;
  int rc = device_info(&di);
  if (rc != ATTN_OK) return rc;
  int status = 0;
  if ((e = cudaMemcpyFromSymbol(&status, g_status, sizeof(int))) != cudaSuccess) return cuda_fail(e);
  if (status != kDevOk) {
    const int zero = 0;
    if ((e = cudaMemcpyToSymbol(g_status, &zero, sizeof(int))) != cudaSuccess) return cuda_fail(e);
    return ATTN_ERR_TIMEOUT;
  }
  return ATTN_OK;
}

const char* attn_status_string(int status) {
  switch (status) {
    case ATTN_OK: return "ok";
    case ATTN_ERR_INVALID_ARG: return "invalid argument";
    case ATTN_ERR_UNSUPPORTED: return "unsupported head size or device";
    case ATTN_ERR_CUDA: return "CUDA error";
    case ATTN_ERR_TIMEOUT: return "a bounded wait inside a kernel timed out";
    case ATTN_ERR_SCRATCH_TOO_SMALL:
      return "these sizes need more scratch than the library's fixed scratch array holds";
    default: return "unknown status";
  }
}

int attn_last_cuda_error(void) { return g_last_cuda_error.load(); }

uint64_t attn_set_wait_limit_ns(uint64_t limit_ns) {
  return g_limit_ns.exchange(limit_ns == 0 ? kDefaultLimitNs : limit_ns);
}

uint64_t attn_launch_count(void) { return g_launches.load(); }

int attn_diag_tile(const void* q, const void* k, const void* p, const void* v, float* s,
                   float* o, struct CUstream_st* stream) {
  if (!q || !k || !p || !v || !s || !o) return ATTN_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(p) || !aligned16(v) || !aligned16(s) ||
      !aligned16(o))
    return ATTN_ERR_INVALID_ARG;
  DeviceInfo* di = nullptr;
  int rc = device_info(&di);
  if (rc != ATTN_OK) return rc;
  CUtensorMap tmq, tmk, tmv;
  if ((rc = encode_2d(&tmq, q)) != ATTN_OK) return rc;
  if ((rc = encode_2d(&tmk, k)) != ATTN_OK) return rc;
  if ((rc = encode_2d(&tmv, v)) != ATTN_OK) return rc;
  cudaError_t e = launch_diag_tile(tmq, tmk, tmv, p, s, o, make_ctx(*di, stream));
  if (e != cudaSuccess) return cuda_fail(e);
  g_launches.fetch_add(1);
  return ATTN_OK;
}

int attn_diag_wait_timeout(uint64_t limit_ns, struct CUstream_st* stream) {
  if (limit_ns == 0 || limit_ns > 10000000000ull) return ATTN_ERR_INVALID_ARG;
  DeviceInfo* di = nullptr;
  int rc = device_info(&di);
  if (rc != ATTN_OK) return rc;
  cudaError_t e = launch_diag_wait_timeout(limit_ns, make_ctx(*di, stream));
  if (e != cudaSuccess) return cuda_fail(e);
  g_launches.fetch_add(1);
  return ATTN_OK;
}

}  // extern "C"
