// Chunk attention on CUDA cores (fp32 arithmetic): the path for fp32
// workloads and for head dims the tensor-core kernel does not take, and the
// step between the oracle and the tensor-core kernel when checking layouts.
//
// "LiveAnimate" 方法: each query token of the current block attends, without
// mask, to every token of its bounded context (static sink, dynamic sink,
// window, the current block itself); ConvKV adds the compressed memory.
//
// A CTA takes kRows query rows of one head and walks the context in tiles
// of kKeys keys, staged in shared memory as fp32 (e4m3 dequantised with the
// slot's scale); the next tile is loaded into registers while the current
// one is computed.  Per slot the query rows are turned by
// (t0_cur + frame - t0_slot, row, col) into shared memory: keys are stored
// turned by their within-block position, so <R(pq) q, R(pk) k> =
// <R(pq - t0_slot) q, R(pk - t0_slot) k> with the second factor exactly the
// stored key.  The 16 threads of a row take 2 scores each (full dot
// products from shared memory), share the running max and sum by xor
// shuffles over those 16 lanes (online softmax, fp32), and each accumulates
// D/16 output dims of P V: dims g*64 + 4c .. g*64 + 4c + 3 for thread c of
// the row, so the row's V reads are contiguous 16-byte loads.
#include "dev_common.cuh"

namespace la {

namespace {

constexpr int kRows = 16;                 // query rows per CTA
constexpr int kKeys = 32;                 // keys per tile
constexpr int kThreads = 256;             // 16 threads per row

template <int D>
struct SimtSmem {
  float q[kRows][D + 1];                  // turned query rows of the current slot (+1: the
                                          // warp's two rows on different banks)
  float k[kKeys][D + 1];                  // +1: a row's 16 threads read 16 keys, no bank conflicts
  __align__(16) float v[kKeys][D];
};

// Element e of row j of a [rows][D] page of dtype dt, as fp32 (scale applied).
__device__ __forceinline__ float page_elem(const char* base, size_t idx, int dt, float scale) {
  if (dt == LA_F32) return reinterpret_cast<const float*>(base)[idx];
  if (dt == LA_BF16) return bf16_bits_to_f32(reinterpret_cast<const uint16_t*>(base)[idx]);
  return e4m3_to_f32(reinterpret_cast<const uint8_t*>(base)[idx]) * scale;
}

template <int D>
__global__ void __launch_bounds__(kThreads) attn_simt_kernel(AttnArgs a) {
  constexpr int kPer = kKeys * D / kThreads;          // tile elements per thread (K and V each)
  constexpr int kDpt = D / 16;                        // output dims per thread
  constexpr int kGroups = kDpt / 4;                   // 4-dim groups, 64 dims apart
  __shared__ __align__(16) SimtSmem<D> sm;
  const int tid = threadIdx.x;
  const int r = tid >> 4, c = tid & 15;               // row in the CTA, position in the row
  const int h = blockIdx.y;
  const int t = blockIdx.x * kRows + r;
  const bool row_ok = t < a.T;
  const DevContext& ctx = *a.ctx;
  const int n_slots = ctx.n_slots;
  if (n_slots < 1 || n_slots > kMaxAttnSlots) {
    if (tid == 0) record_error(a.err, LA_ERR_DEVICE, KID_ATTN_SIMT, n_slots, 0);
    return;
  }
  int f = 0, hh = 0, ww = 0;
  if (row_ok) token_pos(a.rope, t, f, hh, ww);
  // this thread's dims of the row: dim(i) = (i / 4) * 64 + 4c + i % 4
  auto dim = [&](int i) { return (i >> 2) * 64 + 4 * c + (i & 3); };
  // raw query row: kDpt dims per thread, kept in registers
  float q[kDpt];
#pragma unroll
  for (int i = 0; i < kDpt; ++i) {
    const size_t idx = ((size_t)t * a.H + h) * D + dim(i);
    q[i] = row_ok ? page_elem(reinterpret_cast<const char*>(a.q), idx, a.q_dtype, 1.f) : 0.f;
  }
  float m = -INFINITY, l = 0.f, o[kDpt];
#pragma unroll
  for (int i = 0; i < kDpt; ++i) o[i] = 0.f;

  for (int s = 0; s < n_slots; ++s) {
    const int kind = ctx.kind[s], tokens = ctx.tokens[s];
    const char *kb, *vb;
    int rows, kvt = a.kv_dtype;
    float ks = 1.f, vs = 1.f;
    if ((kind == SLOT_FRAME && (ctx.frame[s] < 0 || ctx.frame[s] >= a.n_frames)) ||
        (kind == SLOT_MEMORY && (!a.mem_krot || !a.mem_v)) || kind < 0 || kind > SLOT_MEMORY) {
      if (tid == 0) record_error(a.err, LA_ERR_DEVICE, KID_ATTN_SIMT, kind, ctx.frame[s]);
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
      if (tid == 0) record_error(a.err, LA_ERR_DEVICE, KID_ATTN_SIMT, tokens, rows);
      return;
    }
    const int dtq = ctx.t0_cur + f - ctx.t0[s];
    const bool bad_pos = row_ok && (dtq < 0 || dtq >= a.rope.max_t);
    if (__syncthreads_or(bad_pos)) {
      if (bad_pos) record_error(a.err, LA_ERR_DEVICE, KID_ATTN_SIMT, dtq, s);
      return;
    }
    // this slot's turned query rows into shared memory
#pragma unroll
    for (int p = 0; p < kDpt; p += 2) {
      const int d = dim(p);
      float2 y = make_float2(0.f, 0.f);
      if (row_ok) y = rot_exact(q[p], q[p + 1], rope_cs(a.rope, d, dtq, hh, ww));
      sm.q[r][d] = y.x;
      sm.q[r][d + 1] = y.y;
    }
    const size_t head_off = (size_t)h * rows * D;
    const int n_tiles = (tokens + kKeys - 1) / kKeys;
    float kr[kPer], vr[kPer];
    auto load_tile = [&](int tile) {                  // tile -> registers (fp32)
#pragma unroll
      for (int i = 0; i < kPer; ++i) {
        const int e = i * kThreads + tid;             // element of the tile, key-major
        const int key = tile * kKeys + e / D;
        const size_t idx = head_off + (size_t)key * D + (e % D);
        const bool in = key < tokens;
        kr[i] = in ? page_elem(kb, idx, kvt, ks) : 0.f;
        vr[i] = in ? page_elem(vb, idx, kvt, vs) : 0.f;
      }
    };
    if (n_tiles > 0) load_tile(0);
    for (int tile = 0; tile < n_tiles; ++tile) {
      __syncthreads();                                // previous tile (and q) no longer read
#pragma unroll
      for (int i = 0; i < kPer; ++i) {
        const int e = i * kThreads + tid;
        sm.k[e / D][e % D] = kr[i];
        sm.v[e / D][e % D] = vr[i];
      }
      __syncthreads();
      if (tile + 1 < n_tiles) load_tile(tile + 1);    // in flight during the compute below
      // scores of keys 2c, 2c+1 of this tile
      const int key0 = 2 * c;
      float s0 = 0.f, s1 = 0.f;
#pragma unroll 16
      for (int d = 0; d < D; ++d) {
        const float qd = sm.q[r][d];
        s0 = fmaf(qd, sm.k[key0][d], s0);
        s1 = fmaf(qd, sm.k[key0 + 1][d], s1);
      }
      const int valid = tokens - tile * kKeys;
      s0 = key0 < valid ? s0 * a.scale : -INFINITY;
      s1 = key0 + 1 < valid ? s1 * a.scale : -INFINITY;
      float mx = fmaxf(s0, s1);
#pragma unroll
      for (int o2 = 8; o2; o2 >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o2));
      const float m_new = fmaxf(m, mx);               // finite: key 0 of a tile is always valid
      const float corr = expf(m - m_new);
      const float p0 = expf(s0 - m_new), p1 = expf(s1 - m_new);
      float ps = p0 + p1;
#pragma unroll
      for (int o2 = 8; o2; o2 >>= 1) ps += __shfl_xor_sync(0xffffffffu, ps, o2);
      l = l * corr + ps;
      m = m_new;
#pragma unroll
      for (int i = 0; i < kDpt; ++i) o[i] *= corr;
      // P V: the row's 32 probabilities come from its 16 lanes by shuffles
      const int lane_row = (tid & 31) & ~15;
#pragma unroll 8
      for (int kk = 0; kk < kKeys; ++kk) {
        const float pk = __shfl_sync(0xffffffffu, (kk & 1) ? p1 : p0, lane_row + (kk >> 1));
#pragma unroll
        for (int g = 0; g < kGroups; ++g) {
          const float4 v4 = *reinterpret_cast<const float4*>(&sm.v[kk][g * 64 + 4 * c]);
          o[4 * g] = fmaf(pk, v4.x, o[4 * g]);
          o[4 * g + 1] = fmaf(pk, v4.y, o[4 * g + 1]);
          o[4 * g + 2] = fmaf(pk, v4.z, o[4 * g + 2]);
          o[4 * g + 3] = fmaf(pk, v4.w, o[4 * g + 3]);
        }
      }
    }
    __syncthreads();                                  // q of this slot no longer read
  }
  if (!row_ok) return;
  const float inv_l = 1.f / l;
  const size_t out_off = ((size_t)t * a.H + h) * D;
  if (a.q_dtype == LA_F32) {
    float* p = reinterpret_cast<float*>(a.out) + out_off;
#pragma unroll
    for (int g = 0; g < kGroups; ++g)
      *reinterpret_cast<float4*>(p + g * 64 + 4 * c) =
          make_float4(o[4 * g] * inv_l, o[4 * g + 1] * inv_l, o[4 * g + 2] * inv_l, o[4 * g + 3] * inv_l);
  } else {
    uint16_t* p = reinterpret_cast<uint16_t*>(a.out) + out_off;
#pragma unroll
    for (int g = 0; g < kGroups; ++g)
      *reinterpret_cast<uint2*>(p + g * 64 + 4 * c) =
          make_uint2(pack_bf16x2(o[4 * g] * inv_l, o[4 * g + 1] * inv_l),
                     pack_bf16x2(o[4 * g + 2] * inv_l, o[4 * g + 3] * inv_l));
  }
}

}  // namespace

cudaError_t launch_attn_simt(const AttnArgs& a, cudaStream_t s) {
  if (a.T < 1 || a.H < 1 || a.H > 65535) return cudaErrorInvalidValue;
  dim3 grid((a.T + kRows - 1) / kRows, a.H);
  if (a.D == 128) attn_simt_kernel<128><<<grid, kThreads, 0, s>>>(a);
  else if (a.D == 64) attn_simt_kernel<64><<<grid, kThreads, 0, s>>>(a);
  else return cudaErrorInvalidValue;
  count_launches(1);
  return cudaGetLastError();
}

}  // namespace la
