// attn_fwd_f32.cu -- float32 multi-head scaled dot-product attention forward
// on the CUDA cores.
//
// Same operation as the tensor-core path (eq. (1) of "Attention Is All You
// Need", section 3.2.1, masks of section 3.2.3), for float32 tensors where
// the tensor-core path's bf16 rounding would not meet a 1e-4 tolerance.  One
// thread owns one query row; K/V tiles of 32 keys are staged in shared
// memory and consumed with a streaming softmax in base 2 (scale*log2(e)
// folded into the scores): per tile, the new running max rescales the
// accumulator once, then each key adds 2^(x - m) * v.
#include "attn_internal.cuh"

namespace attn {
namespace {

constexpr int ROWS_PER_CTA = 64;
constexpr int KEYS_PER_TILE = 32;

template <int D>
__global__ void __launch_bounds__(ROWS_PER_CTA)
    attn_fwd_f32_kernel(const float* __restrict__ q, const float* __restrict__ k,
                        const float* __restrict__ v, float* __restrict__ o,
                        float* __restrict__ lse, int H, int n_q, int n_k, float scale_log2,
                        int mask, const int* __restrict__ key_lens) {
  __shared__ float ks[KEYS_PER_TILE][D];
  __shared__ float vs[KEYS_PER_TILE][D];
  const int bh = blockIdx.y;
  const int row0 = blockIdx.x * ROWS_PER_CTA;
  const int row = row0 + threadIdx.x;
  const bool valid = row < n_q;

  int limit = n_k;
  if (mask == kMaskKeyPadding) limit = min(max(key_lens[bh / H], 0), n_k);
  int kend = limit;  // keys this CTA needs
  if (mask == kMaskCausal) kend = min(kend, min(row0 + ROWS_PER_CTA, n_q));

  float qr[D], acc[D];
  const float* qp = q + (static_cast<size_t>(bh) * n_q + (valid ? row : 0)) * D;
#pragma unroll
  for (int t = 0; t < D; ++t) {
    qr[t] = valid ? qp[t] * scale_log2 : 0.f;
    acc[t] = 0.f;
  }
  float m = -INFINITY, l = 0.f;
  const int my_end = mask == kMaskCausal ? min(limit, row + 1) : limit;

  const float* kb = k + static_cast<size_t>(bh) * n_k * D;
  const float* vb = v + static_cast<size_t>(bh) * n_k * D;
  for (int j0 = 0; j0 < kend; j0 += KEYS_PER_TILE) {
    const int nkeys = min(KEYS_PER_TILE, kend - j0);
    for (int e = threadIdx.x; e < KEYS_PER_TILE * D; e += ROWS_PER_CTA) {
      const int jj = e / D, t = e % D;
      const bool in = jj < nkeys;
      ks[jj][t] = in ? kb[static_cast<size_t>(j0 + jj) * D + t] : 0.f;
      vs[jj][t] = in ? vb[static_cast<size_t>(j0 + jj) * D + t] : 0.f;
    }
    __syncthreads();
    if (valid && j0 < my_end) {
      const int nvis = min(nkeys, my_end - j0);
      float x[KEYS_PER_TILE];
      float tmax = -INFINITY;
#pragma unroll
      for (int jj = 0; jj < KEYS_PER_TILE; ++jj) {
        float dot = 0.f;
#pragma unroll
        for (int t = 0; t < D; ++t) dot = fmaf(qr[t], ks[jj][t], dot);
        x[jj] = jj < nvis ? dot : -INFINITY;
        tmax = fmaxf(tmax, x[jj]);
      }
      const float m_new = fmaxf(m, tmax);
      const float alpha = exp2f(m - m_new);  // 0 on the first visible tile
      l *= alpha;
#pragma unroll
      for (int t = 0; t < D; ++t) acc[t] *= alpha;
      m = m_new;
#pragma unroll
      for (int jj = 0; jj < KEYS_PER_TILE; ++jj) {
        const float pj = exp2f(x[jj] - m);
        l += pj;
#pragma unroll
        for (int t = 0; t < D; ++t) acc[t] = fmaf(pj, vs[jj][t], acc[t]);
      }
    }
    __syncthreads();
  }
  if (!valid) return;
  const float inv = l > 0.f ? 1.f / l : 0.f;
  float* op = o + (static_cast<size_t>(bh) * n_q + row) * D;
#pragma unroll
  for (int t = 0; t < D; ++t) op[t] = acc[t] * inv;
  if (lse != nullptr)
    lse[static_cast<size_t>(bh) * n_q + row] =
        l > 0.f ? (m + log2f(l)) * 0.693147180559945309f : -INFINITY;
}

template <int D>
cudaError_t launch_d(const Problem& pb, const LaunchCtx& ctx) {
  dim3 grid((pb.n_q + ROWS_PER_CTA - 1) / ROWS_PER_CTA, pb.B * pb.H);
  attn_fwd_f32_kernel<D><<<grid, ROWS_PER_CTA, 0, ctx.stream>>>(
      static_cast<const float*>(pb.q), static_cast<const float*>(pb.k),
      static_cast<const float*>(pb.v), static_cast<float*>(pb.o), pb.lse, pb.H, pb.n_q,
      pb.n_k, pb.scale * 1.4426950408889634f, pb.mask, pb.key_lens);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_fwd_f32(const Problem& pb, const LaunchCtx& ctx) {
  switch (pb.d) {
    case 16: return launch_d<16>(pb, ctx);
    case 32: return launch_d<32>(pb, ctx);
    case 64: return launch_d<64>(pb, ctx);
    case 128: return launch_d<128>(pb, ctx);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace attn
