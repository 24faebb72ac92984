// Chunk attention on CUDA cores (fp32 arithmetic): the path for fp32
// workloads and for head dims the tensor-core kernel does not take, and the
// step between the oracle and the tensor-core kernel when checking layouts.
//
// "LiveAnimate" 方法: each query token of the current block attends, without
// mask, to every token of its bounded context (static sink, dynamic sink,
// window, the current block itself); ConvKV adds the compressed memory.
//
// One warp per query row, 8 rows (same head) per CTA.  Each lane holds D/32
// dims.  Per slot the query is turned by (t0_cur + frame - t0_slot, row, col):
// keys are stored turned by their within-block position, so
// <R(pq) q, R(pk) k> = <R(pq - t0_slot) q, R(pk - t0_slot) k> with the second
// factor exactly the stored key.  Per key: xor-shuffle dot, online softmax
// (running max, rescaled sum), fp32 accumulation.
#include "dev_common.cuh"

namespace la {

namespace {

template <int DPL>
__device__ __forceinline__ void load_row(const char* base, size_t elem_off, int dtype, float* x) {
  if (dtype == LA_F32) {
    const float* p = reinterpret_cast<const float*>(base) + elem_off;
    if (DPL == 4) {
      float4 u = *reinterpret_cast<const float4*>(p);
      x[0] = u.x; x[1] = u.y; x[2] = u.z; x[3] = u.w;
    } else {
      float2 u = *reinterpret_cast<const float2*>(p);
      x[0] = u.x; x[1] = u.y;
    }
  } else if (dtype == LA_BF16) {
    const uint16_t* p = reinterpret_cast<const uint16_t*>(base) + elem_off;
    if (DPL == 4) {
      uint2 u = *reinterpret_cast<const uint2*>(p);
      x[0] = __uint_as_float(u.x << 16); x[1] = __uint_as_float(u.x & 0xFFFF0000u);
      x[2] = __uint_as_float(u.y << 16); x[3] = __uint_as_float(u.y & 0xFFFF0000u);
    } else {
      uint32_t u = *reinterpret_cast<const uint32_t*>(p);
      x[0] = __uint_as_float(u << 16); x[1] = __uint_as_float(u & 0xFFFF0000u);
    }
  } else {
    const uint8_t* p = reinterpret_cast<const uint8_t*>(base) + elem_off;
#pragma unroll
    for (int i = 0; i < DPL; ++i) x[i] = e4m3_to_f32(p[i]);
  }
}

template <int DPL>
__global__ void __launch_bounds__(256) attn_simt_kernel(AttnArgs a) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int t = blockIdx.x * 8 + warp;
  const int h = blockIdx.y;
  if (t >= a.T) return;
  const DevContext& ctx = *a.ctx;
  int f, hh, ww;
  token_pos(a.rope, t, f, hh, ww);
  const int d0 = lane * DPL;

  float q[DPL];
  load_row<DPL>(reinterpret_cast<const char*>(a.q), ((size_t)t * a.H + h) * a.D + d0, a.q_dtype, q);

  float m = -INFINITY, l = 0.f, o[DPL];
#pragma unroll
  for (int i = 0; i < DPL; ++i) o[i] = 0.f;

  const int n_slots = ctx.n_slots;
  if (n_slots < 1 || n_slots > kMaxAttnSlots) {
    if (lane == 0) record_error(a.err, LA_ERR_DEVICE, KID_ATTN_SIMT, n_slots, 0);
    return;
  }
  for (int s = 0; s < n_slots; ++s) {
    const int kind = ctx.kind[s], tokens = ctx.tokens[s];
    const int dtq = ctx.t0_cur + f - ctx.t0[s];
    if (dtq < 0 || dtq >= a.rope.max_t) {
      if (lane == 0) record_error(a.err, LA_ERR_DEVICE, KID_ATTN_SIMT, dtq, s);
      return;
    }
    float qr[DPL];
#pragma unroll
    for (int p = 0; p < DPL; p += 2) {
      float2 cs = rope_cs(a.rope, d0 + p, dtq, hh, ww);
      float2 y = rot_exact(q[p], q[p + 1], cs);
      qr[p] = y.x;
      qr[p + 1] = y.y;
    }
    const char *kb, *vb;
    int rows;                 // token stride of one head in the source
    int kvt = a.kv_dtype;
    float ks = 1.f, vs = 1.f;
    if ((kind == SLOT_FRAME && (ctx.frame[s] < 0 || ctx.frame[s] >= a.n_frames)) ||
        (kind == SLOT_MEMORY && (!a.mem_krot || !a.mem_v)) || kind < 0 || kind > SLOT_MEMORY) {
      if (lane == 0) record_error(a.err, LA_ERR_DEVICE, KID_ATTN_SIMT, kind, ctx.frame[s]);
      return;
    }
    if (kind == SLOT_FRAME) {
      kb = a.frames + (size_t)ctx.frame[s] * a.G * a.page_stride;
      vb = kb + a.page_stride;
      rows = a.T;
      if (kvt == LA_E4M3) {
        ks = a.frame_scales[((size_t)ctx.frame[s] * 2 + 0) * a.H + h];
        vs = a.frame_scales[((size_t)ctx.frame[s] * 2 + 1) * a.H + h];
      }
    } else if (kind == SLOT_CURRENT) {
      kb = a.cur_k;
      vb = a.cur_v;
      rows = a.T;
      if (kvt == LA_E4M3) { ks = a.cur_scales[h]; vs = a.cur_scales[a.H + h]; }
    } else {
      kb = a.mem_krot;
      vb = a.mem_v;
      rows = a.mem_cap;
      kvt = LA_BF16;
    }
    if (tokens < 0 || tokens > rows) {
      if (lane == 0) record_error(a.err, LA_ERR_DEVICE, KID_ATTN_SIMT, tokens, rows);
      return;
    }
    const float sk = ks * a.scale;
    const size_t head_off = (size_t)h * rows * a.D + d0;
    for (int j = 0; j < tokens; ++j) {
      float k[DPL], v[DPL];
      load_row<DPL>(kb, head_off + (size_t)j * a.D, kvt, k);
      load_row<DPL>(vb, head_off + (size_t)j * a.D, kvt, v);
      float dot = 0.f;
#pragma unroll
      for (int i = 0; i < DPL; ++i) dot = fmaf(qr[i], k[i], dot);
#pragma unroll
      for (int o2 = 16; o2; o2 >>= 1) dot += __shfl_xor_sync(0xffffffffu, dot, o2);
      const float sc = dot * sk;
      const float m_new = fmaxf(m, sc);
      const float corr = expf(m - m_new);
      const float p = expf(sc - m_new);
      l = l * corr + p;
#pragma unroll
      for (int i = 0; i < DPL; ++i) o[i] = o[i] * corr + p * (v[i] * vs);
      m = m_new;
    }
  }
  const float inv_l = 1.f / l;
  float r[DPL];
#pragma unroll
  for (int i = 0; i < DPL; ++i) r[i] = o[i] * inv_l;
  const size_t out_off = ((size_t)t * a.H + h) * a.D + d0;
  if (a.q_dtype == LA_F32) {
    float* p = reinterpret_cast<float*>(a.out) + out_off;
#pragma unroll
    for (int i = 0; i < DPL; ++i) p[i] = r[i];
  } else {
    uint16_t* p = reinterpret_cast<uint16_t*>(a.out) + out_off;
#pragma unroll
    for (int i = 0; i < DPL; i += 2) *reinterpret_cast<uint32_t*>(p + i) = pack_bf16x2(r[i], r[i + 1]);
  }
}

}  // namespace

cudaError_t launch_attn_simt(const AttnArgs& a, cudaStream_t s) {
  dim3 grid((a.T + 7) / 8, a.H);
  if (a.D == 128) attn_simt_kernel<4><<<grid, 256, 0, s>>>(a);
  else if (a.D == 64) attn_simt_kernel<2><<<grid, 256, 0, s>>>(a);
  else return cudaErrorInvalidValue;
  count_launches(1);
  return cudaGetLastError();
}

}  // namespace la
