// attn_internal.cuh -- declarations shared by the library's translation
// units (host launchers and the status codes the kernels record).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <cstdint>

namespace attn {

enum MaskKind : int { kMaskNone = 0, kMaskCausal = 1, kMaskKeyPadding = 2, kMaskBand = 3 };

// Written (first error wins) into the library's device status word.
enum DeviceStatus : int { kDevOk = 0, kDevTimeout = 1 };

// One forward problem, device pointers, [B, H, n, d] contiguous.
struct Problem {
  const void* q;
  const void* k;
  const void* v;
  void* o;
  float* lse;
  int B, H, n_q, n_k, d;
  float scale;
  int mask;
  const int* key_lens;
  int win_left, win_right;  // kMaskBand: query i sees keys i - win_left .. i + win_right
};

// Launch context shared by every launcher.
struct LaunchCtx {
  int num_sms;
  uint64_t limit_ns;  // bounded-wait limit inside kernels
  int* status;        // device address of the status word
  cudaStream_t stream;
};

// Programmatic dependent launch (PTX griddepcontrol): a kernel launched with
// the programmatic stream serialization attribute may start while the kernel
// before it on the stream is still running.  It must pass this wait before it
// touches anything that kernel writes: the wait returns once that grid has
// completed and its memory operations are visible (at once for a kernel
// launched without the attribute).
__device__ __forceinline__ void grid_dependency_wait() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}
// Lets the next kernel on the stream start launching before this grid ends
// (its CTAs still wait in grid_dependency_wait for this grid to complete).
__device__ __forceinline__ void grid_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Launches `kernel` with programmatic stream serialization: it may start (and
// run its prologue) while the previous kernel on the stream drains, so the
// kernel must call grid_dependency_wait() before it reads anything the
// previous kernel writes.  Used only for the second and later kernels of one
// library call, whose predecessor on the stream is always that call's own.
template <typename... KArgs, typename... Args>
inline cudaError_t launch_dependent(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                                   cudaStream_t stream, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<Args&&>(args)...);
}

// tcgen05 bf16 path, d in {16, 32, 64, 128}.  The tensor maps describe Q, K,
// V and O as 3-D (d, n, B*H) bf16 tensors with a (min(d, 64), rows, 1) box
// in the widest swizzle a box row fits (128, 64 or 32 bytes); rows = 128 for
// Q and O, fwd_tc_kv_rows(d) for K and V.
cudaError_t launch_fwd_tc(const Problem& pb, const CUtensorMap& tmq, const CUtensorMap& tmk,
                          const CUtensorMap& tmv, const CUtensorMap& tmo, const LaunchCtx& ctx);
int fwd_tc_kv_rows(int d);

// fp32 SIMT path (d in {16, 32, 64, 128}).
cudaError_t launch_fwd_f32(const Problem& pb, const LaunchCtx& ctx);

// Element strides of a [B, H, n, d] view across batch entries, heads and rows
// (d contiguous).
struct RowStrides {
  long long b, h, n;
};

// Decode path (n_q <= kDecodeMaxQueries new queries against a cache).
constexpr int kDecodeMaxQueries = 8;

struct DecodeProblem {
  const void* q;        // bf16 [B, H, n_q, d]
  const void* k_cache;  // bf16 [B, H, L_max, d]
  const void* v_cache;
  void* o;              // bf16 [B, H, n_q, d]
  float* lse;           // [B, H, n_q] or null
  int B, H, n_q, L_max, d;  // d in {16, 32, 64, 128}
  float scale;
  const int* cache_lens;  // device int32[B] or null (all L_max valid)
  RowStrides sq, sk, sv, so;  // element strides (batch entry, head, row) of q, k, v, o
  int window = -1;  // restricted self-attention: keys [len - 1 - window, len); -1: all keys
};

// How the cache of each head is split across CTAs; workspace_bytes = 0 when
// one CTA per head suffices.
struct DecodePlan {
  int splits;
  int chunk;  // keys per split, a multiple of the 128-key tile
  size_t workspace_bytes;
};
// L_max: the most keys one query sees (the cache length, or the window's).
DecodePlan decode_plan(int B, int H, int n_q, int L_max, int d, int num_sms);
// maps[0..3] (d = 64; unused for the other head sizes, whose kernel reads the
// cache with plain loads): K cache, V cache as 4-D (64, L_max, H, B) bf16 with
// a (64, 128, 1, 1) box, then the same with a (64, 32, 1, 1) box for partial
// last tiles; all with 128-byte swizzle.  workspace holds plan.workspace_bytes.
cudaError_t launch_decode(const DecodeProblem& pb, const CUtensorMap* maps, const DecodePlan& plan,
                          float* workspace, const LaunchCtx& ctx);

// Backward (d = 16, 32 or 64; bf16): gradients of the forward above.
struct BwdProblem {
  const void* q;     // bf16 [B, H, n_q, d]
  const void* k;     // bf16 [B, H, n_k, d]
  const void* v;
  const void* o;     // the forward's output, bf16 [B, H, n_q, d]
  const void* dout;  // dLoss/dO, bf16 [B, H, n_q, d]
  const float* lse;  // the forward's log-sum-exp [B, H, n_q]
  void* dq;          // bf16 outputs, shaped like q, k, v
  void* dk;
  void* dv;
  int B, H, n_q, n_k, d;
  float scale;
  int mask;
  const int* key_lens;
  int win_left, win_right;  // kMaskBand: query i sees keys i - win_left .. i + win_right
  RowStrides so, sdo, sdq;  // strides of o, dout (read with plain loads) and dq (written so)
};

// Workspace of the backward: the per-query constant tiles (one [128 x 16]
// bf16 tile of 4 KB per 128-query tile and head), then the fp32 dQ
// accumulator [B, H, n_q, d].
struct BwdLayout {
  size_t num_qt, cst_off, dq_acc_off, bytes;
};
BwdLayout bwd_layout(int B, int H, int n_q, int d);
bool bwd_head_size_ok(int d);
// maps: Q, K, V, dO as 4-D (d, n, H, B) bf16 with a (d, 128, 1, 1) box; dK,
// dV the same with a (d, 64, 1, 1) box (any strides); the dQ accumulator as 3-D (d, n_q, B*H)
// fp32 with a (min(d, 32), 64, 1) box; each in the swizzle of its box's row
// bytes.  Three launches (preprocess, main, dQ convert).
cudaError_t launch_bwd(const BwdProblem& pb, const CUtensorMap* maps, void* workspace,
                       const LaunchCtx& ctx);

// Diagnostics.  The tensor maps are 2-D (64, 128) bf16, one box each.
cudaError_t launch_diag_tile(const CUtensorMap& tmq, const CUtensorMap& tmk,
                             const CUtensorMap& tmv, const void* p, float* s, float* o,
                             const LaunchCtx& ctx);
cudaError_t launch_diag_wait_timeout(uint64_t limit_ns, const LaunchCtx& ctx);

}  // namespace attn
