// Query rotation for the tensor-core attention (3D RoPE on the query side).
//
// Scores depend only on position differences: <R(pq) q, R(pk) k> =
// <R(pq - t0_s) q, R(pk - t0_s) k>.  Keys sit in the cache turned by their
// within-block position (frame, row, column), so for a slot whose temporal
// base is t0_s the query is turned by (t0_cur + frame - t0_s, row, column)
// and the attention kernel multiplies it with the stored key as is.  This
// kernel writes those per-slot copies for the current block.
#include "dev_common.cuh"
#include "tc_ptx.cuh"

namespace la {

namespace {

using namespace ptx;

constexpr int kTokensPerCta = 16;       // full rows
constexpr int kSplitTokensPerCta = 64;  // split rows

// Loads t0_cur - t0_s of every slot into s_dq and checks that each slot's
// temporal offset stays inside the RoPE table for every frame of the block.
// Called by every thread of the CTA; false (for all of them) on a bad table.
__device__ __forceinline__ bool slot_offsets(const QrotArgs& a, int* s_dq) {
  __shared__ int s_bad;
  const DevContext& ctx = *a.ctx;
  const int n_slots = ctx.n_slots;
  if (n_slots < 1 || n_slots > a.n_qrot || n_slots > kMaxAttnSlots) {
    if (blockIdx.x == 0 && blockIdx.y == 0 && threadIdx.x == 0)
      record_error(a.err, LA_ERR_DEVICE, KID_QROT, n_slots, a.n_qrot);
    return false;
  }
  if (threadIdx.x == 0) s_bad = 0;
  __syncthreads();
  if ((int)threadIdx.x < n_slots) {
    const int s = threadIdx.x;
    const int lo = ctx.t0_cur - ctx.t0[s], hi = lo + a.rope.F - 1;
    s_dq[s] = lo;
    if (lo < 0 || hi >= a.rope.max_t) {
      s_bad = 1;
      if (blockIdx.x == 0 && blockIdx.y == 0) record_error(a.err, LA_ERR_DEVICE, KID_QROT, lo, s);
    }
  }
  __syncthreads();
  return s_bad == 0;
}

// Full rows: qrot[s][h][t] = R(t0_cur + f - t0_s, row, col) q[t][h].
// bf16 cache: bf16 copies.  e4m3 cache: e4m3 codes with one fp32 scale per
// (head, token), qscale[h][t] = m / 448 where m is the largest norm of the
// token's 64 rotation pairs -- rotations keep pair norms, so one scale
// serves every slot and no code saturates.
// Grid: x = tile of 16 tokens, y = head; one thread per 8 dims, the 16
// threads of a token 16 consecutive lanes.  Index math is 32-bit and done
// once per thread; the slot loop only steps the destination and picks the
// table row.
template <bool F8>
__global__ void __launch_bounds__(256) qrot_kernel(QrotArgs a) {
  __shared__ int s_dq[kMaxAttnSlots];                 // t0_cur - t0_s
  if (!slot_offsets(a, s_dq)) return;
  const int n_slots = a.ctx->n_slots;

  const int h = blockIdx.y;
  const int t = blockIdx.x * kTokensPerCta + (threadIdx.x >> 4);
  const int cch = threadIdx.x & 15;
  const bool valid = t < a.T;
  float x[8];
  {
    uint4 u = make_uint4(0u, 0u, 0u, 0u);
    if (valid) u = *reinterpret_cast<const uint4*>(reinterpret_cast<const uint16_t*>(a.q) +
                                                   ((size_t)t * a.H + h) * a.D + cch * 8);
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      x[2 * e] = __uint_as_float(w[e] << 16);
      x[2 * e + 1] = __uint_as_float(w[e] & 0xFFFF0000u);
    }
  }
  float inv = 1.f;
  if (F8) {                                           // all 32 lanes take part
    float n2 = 0.f;
#pragma unroll
    for (int e = 0; e < 4; ++e) n2 = fmaxf(n2, x[2 * e] * x[2 * e] + x[2 * e + 1] * x[2 * e + 1]);
#pragma unroll
    for (int o = 8; o; o >>= 1) n2 = fmaxf(n2, __shfl_xor_sync(0xffffffffu, n2, o));
    const float mn = sqrtf(n2);
    inv = mn > 0.f ? 448.f / mn : 0.f;
    if (valid && cch == 0) a.qscale[(size_t)h * a.T + t] = mn > 0.f ? mn / 448.f : 1.f;
  }
  if (!valid) return;
  int f, hh, ww;
  token_pos(a.rope, t, f, hh, ww);
  // Pairs in the height / width parts turn the same way for every slot:
  // rotate them once.  Only temporal pairs (dims < dt) depend on the slot.
  const int d0 = cch * 8;
  float y[8];
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    y[2 * e] = x[2 * e];
    y[2 * e + 1] = x[2 * e + 1];
    if (d0 + 2 * e >= a.rope.dt) {
      const float2 r = rot_exact(x[2 * e], x[2 * e + 1], rope_cs(a.rope, d0 + 2 * e, 0, hh, ww));
      y[2 * e] = r.x;
      y[2 * e + 1] = r.y;
    }
  }
  const int row_len = a.D;
  const size_t slot_stride = (size_t)a.H * a.T * row_len;
  size_t off = ((size_t)h * a.T + t) * row_len + d0;
  const int pair0 = d0 >> 1, pairs_t = a.rope.dt >> 1;
  // temporal pairs of this chunk: 0..4; with dt a multiple of 4 they come in
  // twos and a table row's pairs sit 16-byte aligned, so (cos, sin) of two
  // pairs is one 16-byte load
  const int np = min(max((a.rope.dt - d0) >> 1, 0), 4);
  const bool vec = (a.rope.dt & 3) == 0;
#pragma unroll 2
  for (int s = 0; s < n_slots; ++s, off += slot_stride) {
    if (np > 0) {
      const float2* row = a.rope.tab_t + (size_t)(s_dq[s] + f) * pairs_t + pair0;
      float2 cs[4];
      if (vec) {
        const float4 c01 = reinterpret_cast<const float4*>(row)[0];
        cs[0] = make_float2(c01.x, c01.y);
        cs[1] = make_float2(c01.z, c01.w);
        if (np > 2) {
          const float4 c23 = reinterpret_cast<const float4*>(row)[1];
          cs[2] = make_float2(c23.x, c23.y);
          cs[3] = make_float2(c23.z, c23.w);
        }
      } else {
#pragma unroll
        for (int e = 0; e < 4; ++e)
          if (e < np) cs[e] = row[e];
      }
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        if (e < np) {
          const float2 r = rot_exact(x[2 * e], x[2 * e + 1], cs[e]);
          y[2 * e] = r.x;
          y[2 * e + 1] = r.y;
        }
      }
    }
    if (F8) {
      uint2 o;
      o.x = cvt_e4m3x4(y[0] * inv, y[1] * inv, y[2] * inv, y[3] * inv);
      o.y = cvt_e4m3x4(y[4] * inv, y[5] * inv, y[6] * inv, y[7] * inv);
      *reinterpret_cast<uint2*>(reinterpret_cast<uint8_t*>(a.qrot) + off) = o;
    } else {
      *reinterpret_cast<uint4*>(reinterpret_cast<uint16_t*>(a.qrot) + off) =
          make_uint4(cvt_bf16x2(y[0], y[1]), cvt_bf16x2(y[2], y[3]), cvt_bf16x2(y[4], y[5]),
                     cvt_bf16x2(y[6], y[7]));
    }
  }
}


// Split rows (bf16, every temporal dim below D/2): each slot gets the first
// half of every row, turned for that slot; the second half, the same for
// every slot, is written once at slot index n_qrot.
// Grid: x = tile of 64 tokens, y = head.  A thread takes 8 dims of each half
// of two neighbouring tokens a, b: it stores their second halves once, then
// their first halves for every slot, so every warp runs the slot loop.
// Tokens a and b normally share a frame, hence a table row: the temporal
// pairs of both then turn together in packed fp32x2,
//   y0 = fma(-x1, s, x0 c),  y1 = fma(x0, s, x1 c),
// with (c, c) and (s, s) from one 16-byte load of the (cos, cos, sin, sin)
// table; a pair that straddles a frame boundary does the same per token.
__device__ __forceinline__ void load_row8(const QrotArgs& a, int t, int h, int d0, float* x) {
  const uint4 u = *reinterpret_cast<const uint4*>(reinterpret_cast<const uint16_t*>(a.q) +
                                                  ((size_t)t * a.H + h) * a.D + d0);
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    x[2 * e] = __uint_as_float(w[e] << 16);
    x[2 * e + 1] = __uint_as_float(w[e] & 0xFFFF0000u);
  }
}
__device__ __forceinline__ void store_row8(void* base, size_t off, const float* y) {
  *reinterpret_cast<uint4*>(reinterpret_cast<uint16_t*>(base) + off) =
      make_uint4(cvt_bf16x2(y[0], y[1]), cvt_bf16x2(y[2], y[3]), cvt_bf16x2(y[4], y[5]),
                 cvt_bf16x2(y[6], y[7]));
}
// Height / width pairs of one token (slot-independent), single roundings.
__device__ __forceinline__ void turn_static(const QrotArgs& a, int t, int d0, const float* x, float* y) {
  int f, hh, ww;
  token_pos(a.rope, t, f, hh, ww);
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    y[2 * e] = x[2 * e];
    y[2 * e + 1] = x[2 * e + 1];
    if (d0 + 2 * e >= a.rope.dt) {
      const float2 r = rot_exact(x[2 * e], x[2 * e + 1], rope_cs(a.rope, d0 + 2 * e, 0, hh, ww));
      y[2 * e] = r.x;
      y[2 * e + 1] = r.y;
    }
  }
}

// The (cos, cos, sin, sin) rows the tile needs -- every slot, the one or
// two frames its 64 tokens fall in -- are staged in shared memory first, so
// the slot loop does not wait on table loads; pair p = 4c + e of a row sits
// at e * 8 + c, so the 8 threads of a token read 8 consecutive entries.
// 4 CTAs per SM (at most 64 registers) keep more Q loads in flight.
constexpr int kStageFrames = 2;
constexpr int kStagePairs = 32;                       // split rows: dt <= D / 2 = 64
__global__ void __launch_bounds__(256, 4) qrot_split_kernel(QrotArgs a) {
  __shared__ int s_dq[kMaxAttnSlots];                 // t0_cur - t0_s
  __shared__ float4 s_tab[kMaxAttnSlots][kStageFrames][kStagePairs];
  if (!slot_offsets(a, s_dq)) return;
  const int n_slots = a.ctx->n_slots;
  const int h = blockIdx.y;
  const int pairs_t = a.rope.dt >> 1;
  const int t_first = blockIdx.x * kSplitTokensPerCta;
  const int f_lo = (int)fdiv((uint32_t)t_first, a.rope.div_hw);
  const int nf = (int)fdiv((uint32_t)min(t_first + kSplitTokensPerCta, a.T) - 1, a.rope.div_hw) - f_lo + 1;
  const bool staged = nf <= kStageFrames && pairs_t <= kStagePairs;
  if (staged) {
    const int per_slot = nf * pairs_t;
    for (int i = threadIdx.x; i < n_slots * per_slot; i += blockDim.x) {
      const int sl = i / per_slot, rem = i - sl * per_slot;
      const int fi = rem / pairs_t, pr = rem - fi * pairs_t;
      s_tab[sl][fi][(pr & 3) * 8 + (pr >> 2)] = a.rope.tab_t2[(size_t)(s_dq[sl] + f_lo + fi) * pairs_t + pr];
    }
  }
  __syncthreads();
  const int ta = t_first + 2 * (threadIdx.x >> 3);
  const int tb = ta + 1;
  if (ta >= a.T) return;
  const bool has_b = tb < a.T;
  const int half = a.D / 2;
  const int d0 = (threadIdx.x & 7) * 8;               // this thread's dims in each half
  const size_t row_a = ((size_t)h * a.T + ta) * half;   // row of token a in one copy
  float xa[8], xb[8], ya[8], yb[8];
  {                                                    // the shared second half, once
    load_row8(a, ta, h, half + d0, xa);
    if (has_b) load_row8(a, tb, h, half + d0, xb);
    load_row8(a, ta, h, d0, ya);                       // first half, loaded early
    if (has_b) load_row8(a, tb, h, d0, yb);
    float za[8], zb[8];
    turn_static(a, ta, half + d0, xa, za);
    const size_t off = (size_t)a.n_qrot * a.H * a.T * half + row_a + d0;
    store_row8(a.qrot, off, za);
    if (has_b) {
      turn_static(a, tb, half + d0, xb, zb);
      store_row8(a.qrot, off + half, zb);
    }
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      xa[e] = ya[e];
      xb[e] = has_b ? yb[e] : 0.f;
    }
  }
  turn_static(a, ta, d0, xa, ya);
  turn_static(a, has_b ? tb : ta, d0, xb, yb);
  const int fa = (int)fdiv((uint32_t)ta, a.rope.div_hw);
  const int fb = has_b ? (int)fdiv((uint32_t)tb, a.rope.div_hw) : fa;
  const int pair0 = d0 >> 1;
  const int np = min(max((a.rope.dt - d0) >> 1, 0), 4);   // temporal pairs here
  // packed (token a, token b) operands of the temporal pairs
  float2 x0[4], x1[4], nx1[4];
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    x0[e] = make_float2(xa[2 * e], xb[2 * e]);
    x1[e] = make_float2(xa[2 * e + 1], xb[2 * e + 1]);
    nx1[e] = make_float2(-xa[2 * e + 1], -xb[2 * e + 1]);
  }
  const size_t slot_stride = (size_t)a.H * a.T * half;
  size_t off = row_a + d0;
#pragma unroll 2
  for (int s = 0; s < n_slots; ++s, off += slot_stride) {
    if (np > 0) {
      if (staged) {
        const float4* ra = &s_tab[s][fa - f_lo][pair0 >> 2];
        const float4* rb = &s_tab[s][fb - f_lo][pair0 >> 2];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          if (e < np) {
            const float4 ca = ra[e * 8], cb = rb[e * 8];
            const float2 y0 = ffma2(nx1[e], make_float2(ca.z, cb.z), fmul2(x0[e], make_float2(ca.x, cb.x)));
            const float2 y1 = ffma2(x0[e], make_float2(ca.z, cb.z), fmul2(x1[e], make_float2(ca.x, cb.x)));
            ya[2 * e] = y0.x; yb[2 * e] = y0.y;
            ya[2 * e + 1] = y1.x; yb[2 * e + 1] = y1.y;
          }
        }
      } else if (fa == fb) {
        const float4* row = a.rope.tab_t2 + (size_t)(s_dq[s] + fa) * pairs_t + pair0;
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          if (e < np) {
            const float4 cs = row[e];
            const float2 c = make_float2(cs.x, cs.y), sn = make_float2(cs.z, cs.w);
            const float2 y0 = ffma2(nx1[e], sn, fmul2(x0[e], c));
            const float2 y1 = ffma2(x0[e], sn, fmul2(x1[e], c));
            ya[2 * e] = y0.x; yb[2 * e] = y0.y;
            ya[2 * e + 1] = y1.x; yb[2 * e + 1] = y1.y;
          }
        }
      } else {                                         // a and b in different frames
        const float2* ra = a.rope.tab_t + (size_t)(s_dq[s] + fa) * pairs_t + pair0;
        const float2* rb = a.rope.tab_t + (size_t)(s_dq[s] + fb) * pairs_t + pair0;
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          if (e < np) {
            const float2 ca = ra[e], cb = rb[e];
            ya[2 * e] = fmaf(-xa[2 * e + 1], ca.y, __fmul_rn(xa[2 * e], ca.x));
            ya[2 * e + 1] = fmaf(xa[2 * e], ca.y, __fmul_rn(xa[2 * e + 1], ca.x));
            yb[2 * e] = fmaf(-xb[2 * e + 1], cb.y, __fmul_rn(xb[2 * e], cb.x));
            yb[2 * e + 1] = fmaf(xb[2 * e], cb.y, __fmul_rn(xb[2 * e + 1], cb.x));
          }
        }
      }
    }
    store_row8(a.qrot, off, ya);
    if (has_b) store_row8(a.qrot, off + half, yb);
  }
}

}  // namespace

cudaError_t launch_qrot(const QrotArgs& a, cudaStream_t s) {
  if (a.D != 128 || a.T < 1 || a.H < 1 || a.H > 65535) return cudaErrorInvalidValue;
  if (a.split && (a.f8 || a.rope.dt > a.D / 2)) return cudaErrorInvalidValue;
  if (a.split && !a.rope.tab_t2) return cudaErrorInvalidValue;
  if (a.split) {
    const dim3 grid((a.T + kSplitTokensPerCta - 1) / kSplitTokensPerCta, a.H);
    qrot_split_kernel<<<grid, 256, 0, s>>>(a);
  } else {
    const dim3 grid((a.T + kTokensPerCta - 1) / kTokensPerCta, a.H);
    if (a.f8)
      qrot_kernel<true><<<grid, 256, 0, s>>>(a);
    else
      qrot_kernel<false><<<grid, 256, 0, s>>>(a);
  }
  count_launches(1);
  return cudaGetLastError();
}

}  // namespace la
