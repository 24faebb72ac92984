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
// rotate: one thread per (head, ring token, 8 channels).
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

__global__ void __launch_bounds__(256) conv_kernel(ConvArgs a) {
  const int chunks = a.D / 8;
  const long long per_tensor = (long long)a.H * a.n_out * chunks;
  const long long total = 2 * per_tensor;
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < total;
       i += (long long)gridDim.x * blockDim.x) {
    int which = (int)(i / per_tensor);                 // 0 = K, 1 = V
    long long r0 = i - which * per_tensor;
    int c = (int)(r0 % chunks);
    long long hj = r0 / chunks;
    int j = (int)(hj % a.n_out);
    int h = (int)(hj / a.n_out);
    const uint16_t* src = reinterpret_cast<const uint16_t*>(which ? a.v : a.kraw) +
                          ((size_t)h * a.T) * a.D + c * 8;
    const uint16_t* w = reinterpret_cast<const uint16_t*>(a.w) +
                        (((size_t)which * a.H + h) * a.D + c * 8) * a.R;
    float acc[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) acc[e] = 0.f;
    for (int r = 0; r < a.R; ++r) {
      int t = a.stride * j + r;
      if (t >= a.T) {
        record_error(a.err, LA_ERR_DEVICE, KID_CONVKV, t, a.T);
        return;
      }
      float x[8];
      load8(src + (size_t)t * a.D, x);
#pragma unroll
      for (int e = 0; e < 8; ++e) acc[e] = fmaf(bf16_bits_to_f32(w[e * a.R + r]), x[e], acc[e]);
    }
    int ri = (a.write0 + j) % a.cap;
    uint16_t* dst = reinterpret_cast<uint16_t*>(which ? a.v_ring : a.k_ring) +
                    ((size_t)h * a.cap + ri) * a.D + c * 8;
    store8(dst, acc);
  }
}

__global__ void __launch_bounds__(256) rotate_ring_kernel(ConvArgs a) {
  const int chunks = a.D / 8;
  const long long total = (long long)a.H * a.n_after * chunks;
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < total;
       i += (long long)gridDim.x * blockDim.x) {
    int c = (int)(i % chunks);
    long long hj = i / chunks;
    int j = (int)(hj % a.n_after);                   // chronological index
    int h = (int)(hj / a.n_after);
    int ri = (a.head_after + j) % a.cap;
    size_t off = ((size_t)h * a.cap + ri) * a.D + c * 8;
    float x[8];
    load8(reinterpret_cast<const uint16_t*>(a.k_ring) + off, x);
#pragma unroll
    for (int p = 0; p < 8; p += 2) {
      int d = c * 8 + p;
      if (d < a.rope.dt) {                             // h = w = 0: only t turns
        float2 cs = a.rope.tab_t[j * (a.rope.dt >> 1) + (d >> 1)];
        float2 y = rot_exact(x[p], x[p + 1], cs);
        x[p] = y.x;
        x[p + 1] = y.y;
      }
    }
    store8(reinterpret_cast<uint16_t*>(a.krot_ring) + off, x);
  }
}

int grid_for(long long work) {
  long long g = (work + 255) / 256;
  if (g > 148LL * 16) g = 148LL * 16;
  return (int)(g < 1 ? 1 : g);
}

}  // namespace

cudaError_t launch_convkv(const ConvArgs& a, cudaStream_t s) {
  long long conv_work = 2LL * a.H * a.n_out * (a.D / 8);
  conv_kernel<<<grid_for(conv_work), 256, 0, s>>>(a);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  long long rot_work = (long long)a.H * a.n_after * (a.D / 8);
  rotate_ring_kernel<<<grid_for(rot_work), 256, 0, s>>>(a);
  count_launches(2);
  return cudaGetLastError();
}

}  // namespace la
