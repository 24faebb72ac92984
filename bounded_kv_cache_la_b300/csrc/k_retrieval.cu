// Pose retrieval for the dynamic sink ("LiveAnimate" 方法: Dynamic Sink keeps
// history blocks retrieved by pose similarity).
//
// One launch per block:
//   1. every CTA builds the query descriptor (17 keypoints, each axis
//      centred by its mean, flattened x0,y0,...) and its inverse norm; CTA 0
//      stores it as table row `pose_row` for later blocks;
//   2. warps score candidates: 8 lanes per candidate, each lane a float4 of
//      the 36-float row (coalesced), fp32 dot, xor-shuffle reduction over
//      the 8 lanes; score = dot * inv|q| * inv|p_j| (0 for zero norm);
//   3. the last CTA to finish ranks the top k+1 under (score desc, id asc)
//      with packed 64-bit keys (orderable score bits << 32 | ~id), a
//      per-thread insertion list and k+1 block-wide arg-max rounds.
#include "dev_common.cuh"

namespace la {

namespace {

constexpr int kThreads = 256;
constexpr int kCandPerCta = 256;   // 8 warps x 4 candidates x 8 iterations

__device__ __forceinline__ uint32_t orderable(float s) {
  uint32_t u = __float_as_uint(s);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float from_orderable(uint32_t o) {
  uint32_t u = (o & 0x80000000u) ? (o & 0x7FFFFFFFu) : ~o;
  return __uint_as_float(u);
}
__device__ __forceinline__ unsigned long long make_key(float s, int id) {
  return ((unsigned long long)orderable(s) << 32) | (unsigned long long)(0xFFFFFFFFu - (uint32_t)id);
}

// Pose descriptor of 17 (x, y) keypoints, one warp: lane l < 17 gets its
// keypoint centred by the per-axis mean, every lane the inverse norm of the
// 34-vector (0 for a zero vector).  Shared by the retrieval and the batch
// history load so that both write bit-identical table rows.
__device__ __forceinline__ void pose_descriptor(float x, float y, int lane, float& cx, float& cy,
                                                float& inv) {
  if (lane >= 17) { x = 0.f; y = 0.f; }
  float sx = x, sy = y;
  for (int o = 16; o; o >>= 1) {
    sx += __shfl_xor_sync(0xffffffffu, sx, o);
    sy += __shfl_xor_sync(0xffffffffu, sy, o);
  }
  cx = x - sx / 17.f;
  cy = y - sy / 17.f;
  if (lane >= 17) { cx = 0.f; cy = 0.f; }
  float ss = cx * cx + cy * cy;
  for (int o = 16; o; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
  inv = ss > 0.f ? 1.0f / sqrtf(ss) : 0.f;
}

__global__ void __launch_bounds__(kThreads) retrieval_kernel(RetrievalArgs a) {
  __shared__ __align__(16) float q[36];
  __shared__ float inv_q;
  __shared__ bool is_last;
  __shared__ unsigned long long red[kThreads / 32];

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

  if (warp == 0) {
    float x = 0.f, y = 0.f;
    if (lane < 17) { x = a.kp[2 * lane]; y = a.kp[2 * lane + 1]; }
    float cx, cy, inv;
    pose_descriptor(x, y, lane, cx, cy, inv);
    if (lane < 17) { q[2 * lane] = cx; q[2 * lane + 1] = cy; }
    if (lane < 2) q[34 + lane] = 0.f;
    if (lane == 0) inv_q = inv;
  }
  __syncthreads();

  if (blockIdx.x == 0 && a.pose_row >= 0) {
    if (a.pose_row >= a.max_history) {
      if (tid == 0) record_error(a.err, LA_ERR_DEVICE, KID_RETRIEVAL, a.pose_row, 0);
    } else if (tid < 36) {
      a.table[(size_t)a.pose_row * 36 + tid] = q[tid];
      if (tid == 0) a.inv_norm[a.pose_row] = inv_q;
    }
  }

  // Scores of this CTA's candidates.
  const int sub = lane & 7;
  const float4 qv = *reinterpret_cast<const float4*>(&q[sub * 4]);
  const float q32 = q[32], q33 = q[33];
  const int cta0 = a.c0 + blockIdx.x * kCandPerCta;
  for (int it = 0; it < kCandPerCta / 32; ++it) {
    int j = cta0 + it * 32 + warp * 4 + (lane >> 3);
    bool ok = j < a.c1;
    float part = 0.f;
    if (ok) {
      const float* row = a.table + (size_t)j * 36;
      float4 p = *reinterpret_cast<const float4*>(row + sub * 4);
      part = p.x * qv.x + p.y * qv.y + p.z * qv.z + p.w * qv.w;
      if (sub == 0) part += row[32] * q32 + row[33] * q33;
    }
    part += __shfl_xor_sync(0xffffffffu, part, 1);
    part += __shfl_xor_sync(0xffffffffu, part, 2);
    part += __shfl_xor_sync(0xffffffffu, part, 4);
    if (ok && sub == 0) a.scores[j] = part * inv_q * a.inv_norm[j];
  }

  // Last CTA ranks.
  __threadfence();
  __syncthreads();
  if (tid == 0) {
    unsigned prev = atomicAdd(&a.topk->done, 1u);
    is_last = (prev == gridDim.x - 1);
  }
  __syncthreads();
  if (!is_last) return;
  __threadfence();

  const int K1 = a.k + 1;                        // rank one extra for the gap
  unsigned long long best[LA_MAX_TOPK + 1];
#pragma unroll
  for (int i = 0; i <= LA_MAX_TOPK; ++i) best[i] = 0ull;
  for (int j = a.c0 + tid; j < a.c1; j += kThreads) {
    unsigned long long key = make_key(__ldcg(a.scores + j), j);
    // insertion into the descending list best[0..K1)
#pragma unroll
    for (int i = 0; i <= LA_MAX_TOPK; ++i) {
      if (i < K1 && key > best[i]) {
        unsigned long long t = best[i];
        best[i] = key;
        key = t;
      }
    }
  }
  int n_found = 0;
  for (int r = 0; r < K1; ++r) {
    unsigned long long m = best[0];
    for (int o = 16; o; o >>= 1) {
      unsigned long long other = __shfl_xor_sync(0xffffffffu, m, o);
      m = other > m ? other : m;
    }
    if (lane == 0) red[warp] = m;
    __syncthreads();
    unsigned long long top = 0ull;
#pragma unroll
    for (int w = 0; w < kThreads / 32; ++w) top = red[w] > top ? red[w] : top;
    __syncthreads();
    if (top == 0ull) break;
    if (best[0] == top) {           // keys are unique (distinct ids): one owner
#pragma unroll
      for (int i = 0; i < LA_MAX_TOPK; ++i) best[i] = best[i + 1];
      best[LA_MAX_TOPK] = 0ull;
    }
    if (tid == 0) {
      a.topk->ids[r] = (int)(0xFFFFFFFFu - (uint32_t)(top & 0xFFFFFFFFull));
      a.topk->scores[r] = from_orderable((uint32_t)(top >> 32));
    }
    ++n_found;
  }
  if (tid == 0) {
    a.topk->n = n_found;
    a.topk->done = 0u;               // ready for the next launch
  }
}

// Batch history load: row i of `table` holds block i's raw keypoints in its
// first 34 floats; one warp per row turns them into the descriptor row (as
// the retrieval kernel writes it) and the inverse norm.
__global__ void __launch_bounds__(256) pose_rows_kernel(float* table, float* inv_norm, int n) {
  const int row = blockIdx.x * 8 + (threadIdx.x >> 5), lane = threadIdx.x & 31;
  if (row >= n) return;                      // whole warps leave together
  float* r = table + (size_t)row * 36;
  float x = 0.f, y = 0.f;
  if (lane < 17) { x = r[2 * lane]; y = r[2 * lane + 1]; }
  float cx, cy, inv;
  pose_descriptor(x, y, lane, cx, cy, inv);  // every lane has read before any writes
  if (lane < 17) { r[2 * lane] = cx; r[2 * lane + 1] = cy; }
  if (lane < 2) r[34 + lane] = 0.f;
  if (lane == 0) inv_norm[row] = inv;
}

}  // namespace

cudaError_t launch_pose_rows(float* table, float* inv_norm, int n, cudaStream_t s) {
  if (n <= 0) return cudaSuccess;
  pose_rows_kernel<<<(n + 7) / 8, 256, 0, s>>>(table, inv_norm, n);
  count_launches(1);
  return cudaGetLastError();
}

cudaError_t launch_retrieval(const RetrievalArgs& a, cudaStream_t s) {
  int n = a.c1 > a.c0 ? a.c1 - a.c0 : 0;
  int grid = n > 0 ? (n + kCandPerCta - 1) / kCandPerCta : 1;
  retrieval_kernel<<<grid, kThreads, 0, s>>>(a);
  count_launches(1);
  return cudaGetLastError();
}

}  // namespace la
