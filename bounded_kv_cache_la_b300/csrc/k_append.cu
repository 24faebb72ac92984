// Cache append: writes a block's K/V from the model layout [T][H][D] into
// cache pages [H][T][D].  Keys are stored already turned by their
// within-block RoPE position (frame, row, column); the slot's temporal base
// is applied later on the query side (score depends only on position
// differences).  ConvKV keeps an un-rotated key copy for its compression.
// An e4m3 cache ("SoulX-LiveAct" 上手实践指南: FP8 KV cache) quantises each
// (head, block) with scale = amax / 448, in two passes (amax, then codes).
//
// One thread moves 16 source bytes (8 bf16 or 4 fp32 values) of one
// (token, head); a CTA covers consecutive tokens of one head, and
// consecutive threads read consecutive 16-byte chunks of a token's row.
#include "dev_common.cuh"

namespace la {

namespace {

template <int SRC>  // LA_F32 or LA_BF16
struct Src;
template <> struct Src<LA_BF16> {
  static constexpr int kVec = 8;
  __device__ static void unpack(const uint4& u, float* x) {
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      x[2 * i] = __uint_as_float(w[i] << 16);
      x[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
    }
  }
  __device__ static void load(const void* base, size_t off, float* x) {
    unpack(*reinterpret_cast<const uint4*>(reinterpret_cast<const uint16_t*>(base) + off), x);
  }
};
template <> struct Src<LA_F32> {
  static constexpr int kVec = 4;
  __device__ static void unpack(const uint4& u, float* x) {
    x[0] = __uint_as_float(u.x); x[1] = __uint_as_float(u.y);
    x[2] = __uint_as_float(u.z); x[3] = __uint_as_float(u.w);
  }
  __device__ static void load(const void* base, size_t off, float* x) {
    unpack(*reinterpret_cast<const uint4*>(reinterpret_cast<const float*>(base) + off), x);
  }
};

template <int VEC>
__device__ __forceinline__ void store_vec(void* base, size_t off, int dtype, const float* x) {
  if (dtype == LA_F32) {
    float* p = reinterpret_cast<float*>(base) + off;
#pragma unroll
    for (int i = 0; i < VEC; i += 4) *reinterpret_cast<float4*>(p + i) = make_float4(x[i], x[i + 1], x[i + 2], x[i + 3]);
  } else {
    uint16_t* p = reinterpret_cast<uint16_t*>(base) + off;
    if (VEC == 8) {
      uint4 u;
      u.x = pack_bf16x2(x[0], x[1]); u.y = pack_bf16x2(x[2], x[3]);
      u.z = pack_bf16x2(x[4], x[5]); u.w = pack_bf16x2(x[6], x[7]);
      *reinterpret_cast<uint4*>(p) = u;
    } else {
      uint2 u;
      u.x = pack_bf16x2(x[0], x[1]); u.y = pack_bf16x2(x[2], x[3]);
      *reinterpret_cast<uint2*>(p) = u;
    }
  }
}

// Within-block rotation of one chunk of VEC dims starting at head dim d0.
template <int VEC>
__device__ __forceinline__ void rotate_chunk(const RopeDims& r, int t, int d0, float* x) {
  int f, hh, ww;
  token_pos(r, t, f, hh, ww);
#pragma unroll
  for (int p = 0; p < VEC; p += 2) {
    float2 cs = rope_cs(r, d0 + p, f, hh, ww);
    float2 y = rot_exact(x[p], x[p + 1], cs);
    x[p] = y.x;
    x[p + 1] = y.y;
  }
}

// Grid: x = token tile (256 / chunks tokens), y = head; one thread per
// chunk of VEC dims.  Reads of a token's head row and writes of the page
// rows stay 16-byte vectors; index math is 32-bit, once per thread.
struct Item {
  int t, h, c;
  bool live;
};
__device__ __forceinline__ Item page_item(const AppendArgs& a, int chunks) {
  const int per_cta = blockDim.x / chunks;
  Item it;
  it.h = blockIdx.y;
  it.t = blockIdx.x * per_cta + (int)threadIdx.x / chunks;
  it.c = (int)threadIdx.x % chunks;
  it.live = it.t < a.T;
  return it;
}

// Values and the raw-key copy keep their dtype, so they move as raw 16-byte
// words; only the key is unpacked, turned and repacked.
template <int SRC>
__global__ void __launch_bounds__(256) append_kernel(AppendArgs a) {
  constexpr int VEC = Src<SRC>::kVec;
  constexpr int ELT = SRC == LA_BF16 ? 2 : 4;
  const Item it = page_item(a, a.D / VEC);
  if (!it.live) return;
  const size_t src_off = ((size_t)it.t * a.H + it.h) * a.D + it.c * VEC;     // [t][h][d]
  const size_t dst_off = ((size_t)it.h * a.T + it.t) * a.D + it.c * VEC;     // [h][t][d]
  const uint4 kw = *reinterpret_cast<const uint4*>(reinterpret_cast<const char*>(a.k) + src_off * ELT);
  const uint4 vw = *reinterpret_cast<const uint4*>(reinterpret_cast<const char*>(a.v) + src_off * ELT);
  float k[VEC];
  Src<SRC>::unpack(kw, k);
  if (a.dst_dtype == SRC) {
    if (a.kraw_dst) *reinterpret_cast<uint4*>(reinterpret_cast<char*>(a.kraw_dst) + dst_off * ELT) = kw;
    *reinterpret_cast<uint4*>(reinterpret_cast<char*>(a.v_dst) + dst_off * ELT) = vw;
  } else {
    float v[VEC];
    Src<SRC>::unpack(vw, v);
    if (a.kraw_dst) store_vec<VEC>(a.kraw_dst, dst_off, a.dst_dtype, k);
    store_vec<VEC>(a.v_dst, dst_off, a.dst_dtype, v);
  }
  rotate_chunk<VEC>(a.rope, it.t, it.c * VEC, k);
  store_vec<VEC>(a.k_dst, dst_off, a.dst_dtype, k);
}

// e4m3 pass 1: per-head amax of the rotated keys and of the values (one
// head per CTA: a warp max, then one shared and one global atomic per warp).
template <int SRC>
__global__ void __launch_bounds__(256) amax_kernel(AppendArgs a) {
  constexpr int VEC = Src<SRC>::kVec;
  const Item it = page_item(a, a.D / VEC);
  float mk = 0.f, mv = 0.f;
  if (it.live) {
    const size_t src_off = ((size_t)it.t * a.H + it.h) * a.D + it.c * VEC;
    float k[VEC], v[VEC];
    Src<SRC>::load(a.k, src_off, k);
    Src<SRC>::load(a.v, src_off, v);
    rotate_chunk<VEC>(a.rope, it.t, it.c * VEC, k);
#pragma unroll
    for (int j = 0; j < VEC; ++j) { mk = fmaxf(mk, fabsf(k[j])); mv = fmaxf(mv, fabsf(v[j])); }
  }
#pragma unroll
  for (int o = 16; o; o >>= 1) {
    mk = fmaxf(mk, __shfl_xor_sync(0xffffffffu, mk, o));
    mv = fmaxf(mv, __shfl_xor_sync(0xffffffffu, mv, o));
  }
  __shared__ unsigned int sm[2];
  if (threadIdx.x < 2) sm[threadIdx.x] = 0u;
  __syncthreads();
  if ((threadIdx.x & 31) == 0) {
    atomicMax(&sm[0], __float_as_uint(mk));
    atomicMax(&sm[1], __float_as_uint(mv));
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    if (sm[0]) atomicMax(&a.amax[it.h], sm[0]);
    if (sm[1]) atomicMax(&a.amax[a.H + it.h], sm[1]);
  }
}

// e4m3 pass 2: code = e4m3_rn_satfinite(x * (448 / amax)), scale = amax / 448.
template <int SRC>
__global__ void __launch_bounds__(256) quant_kernel(AppendArgs a) {
  constexpr int VEC = Src<SRC>::kVec;
  if (blockIdx.x == 0 && blockIdx.y == 0) {
    for (int i = threadIdx.x; i < 2 * a.H; i += blockDim.x) {
      float am = __uint_as_float(a.amax[i]);
      float sc = am > 0.f ? __fdiv_rn(am, 448.f) : 1.f;
      if (i < a.H) a.k_scale[i] = sc; else a.v_scale[i - a.H] = sc;
    }
  }
  const Item it = page_item(a, a.D / VEC);
  if (!it.live) return;
  const int h = it.h;
  const size_t src_off = ((size_t)it.t * a.H + h) * a.D + it.c * VEC;
  const size_t dst_off = ((size_t)h * a.T + it.t) * a.D + it.c * VEC;
  float k[VEC], v[VEC];
  Src<SRC>::load(a.k, src_off, k);
  Src<SRC>::load(a.v, src_off, v);
  rotate_chunk<VEC>(a.rope, it.t, it.c * VEC, k);
  float amk = __uint_as_float(a.amax[h]), amv = __uint_as_float(a.amax[a.H + h]);
  float ik = amk > 0.f ? __fdiv_rn(448.f, amk) : 0.f;
  float iv = amv > 0.f ? __fdiv_rn(448.f, amv) : 0.f;
  uint8_t ck[VEC], cv[VEC];
#pragma unroll
  for (int j = 0; j < VEC; ++j) {
    ck[j] = f32_to_e4m3(__fmul_rn(k[j], ik));
    cv[j] = f32_to_e4m3(__fmul_rn(v[j], iv));
  }
  uint8_t* pk = reinterpret_cast<uint8_t*>(a.k_dst) + dst_off;
  uint8_t* pv = reinterpret_cast<uint8_t*>(a.v_dst) + dst_off;
  if (VEC == 8) {
    uint2 uk, uv;
    uk.x = ck[0] | (ck[1] << 8) | (ck[2] << 16) | ((uint32_t)ck[3] << 24);
    uk.y = ck[4] | (ck[5] << 8) | (ck[6] << 16) | ((uint32_t)ck[7] << 24);
    uv.x = cv[0] | (cv[1] << 8) | (cv[2] << 16) | ((uint32_t)cv[3] << 24);
    uv.y = cv[4] | (cv[5] << 8) | (cv[6] << 16) | ((uint32_t)cv[7] << 24);
    *reinterpret_cast<uint2*>(pk) = uk;
    *reinterpret_cast<uint2*>(pv) = uv;
  } else {
    *reinterpret_cast<uint32_t*>(pk) = ck[0] | (ck[1] << 8) | (ck[2] << 16) | ((uint32_t)ck[3] << 24);
    *reinterpret_cast<uint32_t*>(pv) = cv[0] | (cv[1] << 8) | (cv[2] << 16) | ((uint32_t)cv[3] << 24);
  }
}

}  // namespace

cudaError_t launch_append(const AppendArgs& a, cudaStream_t s) {
  const int vec = a.src_dtype == LA_BF16 ? 8 : 4;
  const int chunks = a.D / vec;                       // 8, 16 or 32: divides 256
  if (a.D % vec || 256 % chunks || a.H < 1 || a.H > 65535 || a.T < 1) return cudaErrorInvalidValue;
  const dim3 grid((a.T + 256 / chunks - 1) / (256 / chunks), a.H);
  if (a.dst_dtype == LA_E4M3) {
    cudaError_t e = cudaMemsetAsync(a.amax, 0, sizeof(unsigned int) * 2 * a.H, s);
    if (e != cudaSuccess) return e;
    if (a.src_dtype == LA_BF16) {
      amax_kernel<LA_BF16><<<grid, 256, 0, s>>>(a);
      quant_kernel<LA_BF16><<<grid, 256, 0, s>>>(a);
    } else {
      amax_kernel<LA_F32><<<grid, 256, 0, s>>>(a);
      quant_kernel<LA_F32><<<grid, 256, 0, s>>>(a);
    }
  } else if (a.src_dtype == LA_BF16) {
    append_kernel<LA_BF16><<<grid, 256, 0, s>>>(a);
  } else {
    append_kernel<LA_F32><<<grid, 256, 0, s>>>(a);
  }
  count_launches(a.dst_dtype == LA_E4M3 ? 2 : 1);
  return cudaGetLastError();
}

}  // namespace la
