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

// Per-slot rotated copies of the queries: qrot[s][h][t] = R(t0_cur + f - t0_s, row, col) q[t][h].
// bf16 cache: bf16 copies.  e4m3 cache: e4m3 codes with one fp32 scale per
// (head, token), qscale[h][t] = m / 448 where m is the largest norm of the
// token's 64 rotation pairs -- rotations keep pair norms, so one scale
// serves every slot and no code saturates.  One thread per 8 dims; the 16
// threads of a (token, head) are 16 consecutive lanes.
template <bool F8>
__global__ void __launch_bounds__(256) qrot_kernel(QrotArgs a) {
  const DevContext& ctx = *a.ctx;
  const int n_slots = ctx.n_slots;
  if (n_slots < 1 || n_slots > a.n_qrot) {
    if (blockIdx.x == 0 && threadIdx.x == 0) record_error(a.err, LA_ERR_DEVICE, KID_QROT, n_slots, a.n_qrot);
    return;
  }
  // every slot's temporal offset must stay inside the RoPE table for every
  // frame of the block (checked up front so that all threads leave together)
  for (int s = 0; s < n_slots; ++s) {
    const int lo = ctx.t0_cur - ctx.t0[s], hi = lo + a.rope.F - 1;
    if (lo < 0 || hi >= a.rope.max_t) {
      if (blockIdx.x == 0 && threadIdx.x == 0) record_error(a.err, LA_ERR_DEVICE, KID_QROT, lo, s);
      return;
    }
  }
  const int chunks = a.D / 8;
  const long long total = (long long)a.T * a.H * chunks;
  const long long stride = (long long)gridDim.x * blockDim.x;
  // warp-uniform trip count (the e4m3 path reduces over 16-lane groups)
  for (long long base = blockIdx.x * (long long)blockDim.x + (threadIdx.x & ~31); base < total;
       base += stride) {
    const long long idx = base + (threadIdx.x & 31);
    const bool valid = idx < total;
    const long long vi = valid ? idx : 0;
    // consecutive threads: dims, then tokens of one head, so each slot copy
    // ([slot][head][token][dim]) is written in long contiguous runs
    const int cch = (int)(vi % chunks);
    const long long ht = vi / chunks;
    const int t = (int)(ht % a.T);
    const int h = (int)(ht / a.T);
    const size_t th = (size_t)t * a.H + h;
    uint4 u = *reinterpret_cast<const uint4*>(reinterpret_cast<const uint16_t*>(a.q) + th * a.D + cch * 8);
    float x[8];
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      x[2 * e] = __uint_as_float(w[e] << 16);
      x[2 * e + 1] = __uint_as_float(w[e] & 0xFFFF0000u);
    }
    float inv = 1.f;
    if (F8) {
      float n2 = 0.f;
#pragma unroll
      for (int e = 0; e < 4; ++e) n2 = fmaxf(n2, x[2 * e] * x[2 * e] + x[2 * e + 1] * x[2 * e + 1]);
#pragma unroll
      for (int o = 8; o; o >>= 1) n2 = fmaxf(n2, __shfl_xor_sync(0xffffffffu, n2, o));
      const float mn = sqrtf(n2);
      inv = mn > 0.f ? 448.f / mn : 0.f;
      if (valid && cch == 0) a.qscale[(size_t)h * a.T + t] = mn > 0.f ? mn / 448.f : 1.f;
    }
    if (!valid) continue;
    int f, hh, ww;
    token_pos(a.rope, t, f, hh, ww);
    // Pairs in the height / width parts turn the same way for every slot:
    // rotate them once.  Only temporal pairs (dims < dt) depend on the slot.
    const int d0 = cch * 8;
    float y[8];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      if (d0 + 2 * e >= a.rope.dt) {
        const float2 r = rot_exact(x[2 * e], x[2 * e + 1], rope_cs(a.rope, d0 + 2 * e, 0, hh, ww));
        y[2 * e] = r.x;
        y[2 * e + 1] = r.y;
      }
    }
    const bool temporal = d0 < a.rope.dt;
    uint4 fixed_bf16{};
    uint2 fixed_f8{};
    if (!temporal) {
      if (F8) {
        fixed_f8.x = cvt_e4m3x4(y[0] * inv, y[1] * inv, y[2] * inv, y[3] * inv);
        fixed_f8.y = cvt_e4m3x4(y[4] * inv, y[5] * inv, y[6] * inv, y[7] * inv);
      } else {
        fixed_bf16 = make_uint4(cvt_bf16x2(y[0], y[1]), cvt_bf16x2(y[2], y[3]), cvt_bf16x2(y[4], y[5]),
                                cvt_bf16x2(y[6], y[7]));
      }
    }
    for (int s = 0; s < n_slots; ++s) {
      const size_t off = (((size_t)s * a.H + h) * a.T + t) * a.D + d0;
      if (!temporal) {
        if (F8)
          *reinterpret_cast<uint2*>(reinterpret_cast<uint8_t*>(a.qrot) + off) = fixed_f8;
        else
          *reinterpret_cast<uint4*>(reinterpret_cast<uint16_t*>(a.qrot) + off) = fixed_bf16;
        continue;
      }
      const int dtq = ctx.t0_cur + f - ctx.t0[s];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        if (d0 + 2 * e < a.rope.dt) {
          const float2 r = rot_exact(x[2 * e], x[2 * e + 1], a.rope.tab_t[dtq * (a.rope.dt >> 1) + ((d0 + 2 * e) >> 1)]);
          y[2 * e] = r.x;
          y[2 * e + 1] = r.y;
        }
      }
      if (F8) {
        uint2 o;
        o.x = cvt_e4m3x4(y[0] * inv, y[1] * inv, y[2] * inv, y[3] * inv);
        o.y = cvt_e4m3x4(y[4] * inv, y[5] * inv, y[6] * inv, y[7] * inv);
        *reinterpret_cast<uint2*>(reinterpret_cast<uint8_t*>(a.qrot) + off) = o;
      } else {
        uint4 o;
        o.x = cvt_bf16x2(y[0], y[1]);
        o.y = cvt_bf16x2(y[2], y[3]);
        o.z = cvt_bf16x2(y[4], y[5]);
        o.w = cvt_bf16x2(y[6], y[7]);
        *reinterpret_cast<uint4*>(reinterpret_cast<uint16_t*>(a.qrot) + off) = o;
      }
    }
  }
}

}  // namespace

cudaError_t launch_qrot(const QrotArgs& a, cudaStream_t s) {
  if (a.D != 128) return cudaErrorInvalidValue;
  long long work = (long long)a.T * a.H * (a.D / 8);
  long long grid = (work + 255) / 256;
  if (grid > 148LL * 16) grid = 148LL * 16;
  if (a.f8)
    qrot_kernel<true><<<(int)grid, 256, 0, s>>>(a);
  else
    qrot_kernel<false><<<(int)grid, 256, 0, s>>>(a);
  count_launches(1);
  return cudaGetLastError();
}

}  // namespace la
