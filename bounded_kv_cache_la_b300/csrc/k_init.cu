// RoPE cos/sin tables, built once per cache in fp64 and stored as fp32.
#include "dev_common.cuh"

namespace la {

// tab[pos][i] = (cos, sin)(pos * theta^(-2i/d_axis)) for one axis part of the
// 3D RoPE (t, h or w).
__global__ void init_axis_table(float2* tab, int rows, int d_axis, double theta) {
  int half = d_axis >> 1;
  int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (half == 0 || i >= rows * half) return;
  int pos = i / half;
  int p = i - pos * half;
  double freq = pow(theta, (-2.0 * p) / d_axis);
  double ang = (double)pos * freq;
  tab[i] = make_float2((float)cos(ang), (float)sin(ang));
}

// tab2[i] = (cos, cos, sin, sin) of tab[i]: one 16-byte load gives the
// packed (c, c) and (s, s) operands that turn two tokens at once.
__global__ void dup_table(float4* tab2, const float2* tab, int n) {
  int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= n) return;
  const float2 cs = tab[i];
  tab2[i] = make_float4(cs.x, cs.x, cs.y, cs.y);
}

cudaError_t launch_init_tables(float2* tab_t, int max_t, int dt, float2* tab_h, int GH, int dh,
                               float2* tab_w, int GW, int dw, double theta, float4* tab_t2,
                               cudaStream_t s) {
  struct { float2* p; int rows; int d; } parts[3] = {{tab_t, max_t, dt}, {tab_h, GH, dh},
                                                     {tab_w, GW, dw}};
  for (auto& pt : parts) {
    int n = pt.rows * (pt.d / 2);
    if (n <= 0) continue;
    init_axis_table<<<(n + 255) / 256, 256, 0, s>>>(pt.p, pt.rows, pt.d, theta);
    count_launches(1);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  const int n_t = max_t * (dt / 2);
  if (tab_t2 && n_t > 0) {
    dup_table<<<(n_t + 255) / 256, 256, 0, s>>>(tab_t2, tab_t, n_t);
    count_launches(1);
    return cudaGetLastError();
  }
  return cudaSuccess;
}

}  // namespace la
