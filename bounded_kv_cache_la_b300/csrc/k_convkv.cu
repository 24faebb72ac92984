// ConvKV memory update ("SoulX-LiveAct" 技术内核: older K/V compressed by a 1D
// convolution, ratio 5:1, into fixed-length memory with RoPE positions reset).
//
// On eviction of one exact block, for each head h, channel c and output j:
//   m[j][h][c] = sum_{r < R} w[h][c][r] * x[stride*j + r][h][c]      (fp32, bf16 out)
// for the raw keys and for the values (separate weights).  The memory is a
// per-head ring of `cap` tokens holding the newest compressed tokens; the
// rotated-key ring is then rebuilt so that the token j-th oldest carries the
// temporal position j (h = w = 0), which is what "positions reset" means here.
//
// conv: one thread per (K/V, head, output token, 8 channels); the 5 input
// rows are 16-byte loads along the channel axis (coalesced across threads).
// rotate: one thread per (head, ring token, 8 channels).  A CTA covers
// consecutive tokens of one head; index math is 32-bit, once per thread.
#include "dev_common.cuh"

namespace la {

namespace {

__device__ __forceinline__ void load8(const uint16_t* p, float* x) {
  uint4 u = *reinterpret_cast<const uint4*>(p);
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    x[2 * i] = __uint_as_float(w[i] << 16);
    x[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
  }
}
__device__ __forceinline__ void store8(uint16_t* p, const float* x) {
  uint4 u;
  u.x = pack_bf16x2(x[0], x[1]); u.y = pack_bf16x2(x[2], x[3]);
  u.z = pack_bf16x2(x[4], x[5]); u.w = pack_bf16x2(x[6], x[7]);
  *reinterpret_cast<uint4*>(p) = u;
}

// Grid: x = output-token tile (256 / chunks tokens), y = (K/V, head); one
// thread per 8 channels.  RK > 0: kernel size known at compile time, loops
// unrolled and the 8 x RK weights of a thread (contiguous, 16 * RK bytes)
// read with 16-byte loads; RK = 0: any kernel size, weights read per tap.
template <int RK>
__global__ void __launch_bounds__(256) conv_kernel(ConvArgs a) {
  const int R = RK > 0 ? RK : a.R;
  const int chunks = a.D / 8;
  const int which = (int)blockIdx.y >= a.H ? 1 : 0;  // 0 = K, 1 = V
  const int h = (int)blockIdx.y - which * a.H;
  const int j = blockIdx.x * (blockDim.x / chunks) + (int)threadIdx.x / chunks;
  const int c = (int)threadIdx.x % chunks;
  if (j >= a.n_out) return;
  if (a.stride * j + R > a.T) {                        // the last tap must be in the block
    record_error(a.err, LA_ERR_DEVICE, KID_CONVKV, a.stride * j + R - 1, a.T);
    return;
  }
  const uint16_t* src = reinterpret_cast<const uint16_t*>(which ? a.v : a.kraw) +
                        ((size_t)h * a.T + (size_t)a.stride * j) * a.D + c * 8;
  const uint16_t* w = reinterpret_cast<const uint16_t*>(a.w) +
                      (((size_t)which * a.H + h) * a.D + c * 8) * R;
  float acc[8];
#pragma unroll
  for (int e = 0; e < 8; ++e) acc[e] = 0.f;
  if constexpr (RK > 0) {
    // weights of channels c*8 .. c*8+7, taps 0..RK-1: 8 * RK bf16 in a row
    uint4 wq[RK];
#pragma unroll
    for (int q = 0; q < RK; ++q) wq[q] = reinterpret_cast<const uint4*>(w)[q];
    const uint16_t* wv = reinterpret_cast<const uint16_t*>(wq);
    float x[RK][8];
#pragma unroll
    for (int r = 0; r < RK; ++r) load8(src + (size_t)r * a.D, x[r]);
#pragma unroll
    for (int r = 0; r < RK; ++r)
#pragma unroll
      for (int e = 0; e < 8; ++e) acc[e] = fmaf(bf16_bits_to_f32(wv[e * RK + r]), x[r][e], acc[e]);
  } else {
    for (int r = 0; r < R; ++r) {
      float x[8];
      load8(src + (size_t)r * a.D, x);
#pragma unroll
      for (int e = 0; e < 8; ++e) acc[e] = fmaf(bf16_bits_to_f32(w[e * R + r]), x[e], acc[e]);
    }
  }
  int ri = a.write0 + j;
  if (ri >= a.cap) ri -= a.cap;                        // write0 < cap and j < n_out <= cap
  uint16_t* dst = reinterpret_cast<uint16_t*>(which ? a.v_ring : a.k_ring) +
                  ((size_t)h * a.cap + ri) * a.D + c * 8;
  store8(dst, acc);
}

// Grid: x = memory-token tile, y = head; one thread per 8 dims.
__global__ void __launch_bounds__(256) rotate_ring_kernel(ConvArgs a) {
  const int chunks = a.D / 8;
  const int h = blockIdx.y;
  const int j = blockIdx.x * (blockDim.x / chunks) + (int)threadIdx.x / chunks;   // chronological index
  const int c = (int)threadIdx.x % chunks;
  if (j >= a.n_after) return;
  int ri = a.head_after + j;
  if (ri >= a.cap) ri -= a.cap;                        // head_after < cap and j < n_after <= cap
  const size_t off = ((size_t)h * a.cap + ri) * a.D + c * 8;
  float x[8];
  load8(reinterpret_cast<const uint16_t*>(a.k_ring) + off, x);
#pragma unroll
  for (int p = 0; p < 8; p += 2) {
    int d = c * 8 + p;
    if (d < a.rope.dt) {                               // h = w = 0: only t turns
      float2 cs = a.rope.tab_t[j * (a.rope.dt >> 1) + (d >> 1)];
      float2 y = rot_exact(x[p], x[p + 1], cs);
      x[p] = y.x;
      x[p + 1] = y.y;
    }
  }
  store8(reinterpret_cast<uint16_t*>(a.krot_ring) + off, x);
}

}  // namespace

cudaError_t launch_convkv(const ConvArgs& a, cudaStream_t s) {
  const int chunks = a.D / 8;
  if (a.D % 8 || 256 % chunks || a.H < 1 || 2 * a.H > 65535 || a.n_out < 1 || a.n_out > a.cap ||
      a.write0 < 0 || a.write0 >= a.cap || a.n_after < 0 || a.n_after > a.cap || a.head_after < 0 ||
      a.head_after >= a.cap)
    return cudaErrorInvalidValue;
  const int per_cta = 256 / chunks;
  // the 16-byte weight loads need a 16-byte aligned weight tensor
  const dim3 conv_grid((a.n_out + per_cta - 1) / per_cta, 2 * a.H);
  if (a.R == 5 && (reinterpret_cast<uintptr_t>(a.w) & 15) == 0)
    conv_kernel<5><<<conv_grid, 256, 0, s>>>(a);
  else
    conv_kernel<0><<<conv_grid, 256, 0, s>>>(a);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  int launched = 1;
  if (a.n_after > 0) {
    const dim3 rot_grid((a.n_after + per_cta - 1) / per_cta, a.H);
    rotate_ring_kernel<<<rot_grid, 256, 0, s>>>(a);
    ++launched;
  }
  count_launches(launched);
  return cudaGetLastError();
}

}  // namespace la
