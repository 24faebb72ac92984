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

cudaError_t launch_init_tables(float2* tab_t, int max_t, int dt, float2* tab_h, int GH, int dh,
                               float2* tab_w, int GW, int dw, double theta, cudaStream_t s) {
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
  return cudaSuccess;
}

}  // namespace la
