// Internal declarations shared by the host state machine (la_cache.cu) and
// the kernels.  Not part of the public ABI (include/la_cache.h).
#pragma once

#include <cuda_runtime.h>
#include <cuda.h>
#include <stddef.h>
#include <stdint.h>

#include "la_cache.h"

namespace la {

constexpr int kMaxExact = LA_MAX_SLOTS;   // exact slots (cached blocks + current)
constexpr int kMaxAttnSlots = kMaxExact + 1;  // + ConvKV memory slot

enum SlotKind : int { SLOT_FRAME = 0, SLOT_CURRENT = 1, SLOT_MEMORY = 2 };

// Device error word.  code: 0 ok, LA_ERR_DEVICE or LA_ERR_TIMEOUT; the first
// fault wins (atomicCAS on code).
struct DevError {
  int code;
  int kernel;   // KernelId
  int detail0;
  int detail1;
};
enum KernelId : int {
  KID_RETRIEVAL = 1, KID_APPEND = 2, KID_CONVKV = 3, KID_ATTN_SIMT = 4, KID_ATTN_TC = 5,
  KID_QROT = 6, KID_INIT = 7
};

// Slot table of the block being generated.  Written by the host at select,
// read by every attention kernel of the block.
struct DevContext {
  int n_slots;                     // attention slots (memory + exact)
  int kv_len;
  int t0_cur;                      // temporal base of the current block
  int block;
  int kind[kMaxAttnSlots];
  int frame[kMaxAttnSlots];        // frame index for SLOT_FRAME, else -1
  int tokens[kMaxAttnSlots];
  int t0[kMaxAttnSlots];
};

// Retrieval results (top k+1 in descending order).
struct DevTopk {
  unsigned int done;               // CTA completion counter (reset by the last CTA)
  int n;                           // entries written (<= k + 1)
  int ids[LA_MAX_TOPK + 1];
  float scores[LA_MAX_TOPK + 1];
};

// Byte offsets of every region inside the caller's pool.
struct Layout {
  size_t err, ctx, topk;           // control
  size_t ctx_final;                // slot table whose current slot is the block's own frame
  size_t amax;                     // e4m3 amax scratch [2][H] uint32
  size_t pose_tab;                 // [max_history][36] fp32
  size_t inv_norm;                 // [max_history] fp32
  size_t scores;                   // retrieval scratch [max_history] fp32
  size_t rope_t, rope_h, rope_w;   // float2 (cos, sin) tables
  size_t scales;                   // e4m3 [L][n_frames][2][H] fp32
  size_t cur_scales;               // e4m3 [2][H] fp32
  size_t frames;                   // [L][n_frames][G] pages
  size_t cur_pages;                // 2 pages: current block K', V
  size_t qrot;                     // [S][H][T][D] rotated queries (tensor path), kv dtype
  size_t rope_t2;                  // bf16 tensor path: temporal table as (cos, cos, sin, sin)
  size_t ctx_inject;               // slot table of an injected failure (la_debug_inject)
  size_t qscale;                   // e4m3 tensor path: [H][T] fp32 query scales
  size_t sched;                    // tensor path: work items per CTA (attn_tc_schedule)
  size_t part_o, part_ml;          // tensor path, odd query-tile count: pieces' partial results
  size_t mem;                      // ConvKV [L][3][H][cap][D] bf16 (raw K, V, rotated K)
  size_t total;
  size_t page_bytes;               // H * T * D * elt(kv_dtype)
  size_t page_stride;              // page_bytes rounded up to 1024
  int G;                           // pages per frame: 2 (K', V) or 3 (+ raw K)
  int n_frames;                    // frames per layer
  int max_t;                       // rows of the temporal RoPE table
  int n_qrot;                      // rotated-query slots held
  int T;
};

// Division by a run-time constant d >= 1, for numerators below 2^31, as a
// multiply-high, an add and a shift (Granlund and Montgomery, "Division by
// invariant integers using multiplication", 1994): with l = ceil(log2 d) and
// m = floor(2^32 (2^l - d) / d) + 1, n / d = (umulhi(n, m) + n) >> l.
struct FastDiv {
  uint32_t d, m, l;
};
inline FastDiv make_fastdiv(uint32_t d) {
  uint32_t l = 0;
  while ((1ull << l) < d) ++l;
  const uint64_t m = ((1ull << 32) * ((1ull << l) - d)) / d + 1;
  return FastDiv{d, (uint32_t)m, l};
}

struct RopeDims {
  int dt, dh, dw;                  // dims per axis
  int F, GH, GW;                   // block grid
  FastDiv div_hw, div_w;           // by GH * GW and by GW (token -> frame, row, column)
  int max_t;                       // rows of tab_t
  const float2* tab_t;             // [max_t][dt/2]
  const float4* tab_t2;            // [max_t][dt/2] (cos, cos, sin, sin), or null
  const float2* tab_h;             // [GH][dh/2]
  const float2* tab_w;             // [GW][dw/2]
};

// Kernel launches enqueued by the library (every launcher adds its count).
void count_launches(int n);

// ------------------------------------------------------------ kernel launches
// Each returns the cudaError_t of its launch(es).
cudaError_t launch_init_tables(float2* tab_t, int max_t, int dt, float2* tab_h, int GH, int dh,
                               float2* tab_w, int GW, int dw, double theta, float4* tab_t2,
                               cudaStream_t s);

struct RetrievalArgs {
  float kp[34];
  int pose_row;        // table row for the query descriptor, -1 = none
  int c0, c1;          // candidate ids [c0, c1)
  int k;               // picks (<= LA_MAX_TOPK); k + 1 are ranked
  int max_history;
  float* table;        // [max_history][36]
  float* inv_norm;
  float* scores;
  DevTopk* topk;
  DevError* err;
};
cudaError_t launch_retrieval(const RetrievalArgs& a, cudaStream_t s);
// Rows 0..n-1 of `table` hold raw keypoints (34 floats each): turned into
// descriptor rows and inverse norms in place.
cudaError_t launch_pose_rows(float* table, float* inv_norm, int n, cudaStream_t s);

struct AppendArgs {
  const void* k;       // [T][H][D] src_dtype
  const void* v;
  void* k_dst;         // [H][T][D] dst_dtype, RoPE'd by the within-block position
  void* v_dst;
  void* kraw_dst;      // optional [H][T][D] un-rotated copy (ConvKV)
  float* k_scale;      // e4m3: [H]
  float* v_scale;
  unsigned int* amax;  // e4m3 scratch [2][H]
  int T, H, D;
  int src_dtype, dst_dtype;
  RopeDims rope;
  DevError* err;
};
cudaError_t launch_append(const AppendArgs& a, cudaStream_t s);

struct ConvArgs {
  const void* kraw;    // evicted block [H][T][D] bf16
  const void* v;
  const void* w;       // [2][H][D][R] bf16
  void* k_ring;        // [H][cap][D] bf16
  void* v_ring;
  void* krot_ring;
  int T, H, D, R, stride, n_out, cap;
  int write0;          // ring index of the first new token
  int n_after, head_after;   // memory tokens and oldest ring index after the append
  RopeDims rope;
  DevError* err;
};
cudaError_t launch_convkv(const ConvArgs& a, cudaStream_t s);

struct AttnArgs {
  const void* q;       // [T][H][D] q_dtype
  void* out;           // [T][H][D] q_dtype
  int T, H, D, q_dtype, kv_dtype;
  const DevContext* ctx;
  const char* frames;  // layer's first frame page
  size_t page_stride;
  int G;
  int n_frames;        // frames per layer (bound of ctx->frame)
  const char* cur_k;   // current block pages
  const char* cur_v;
  const float* frame_scales;  // e4m3: this layer's [n_frames][2][H]
  const float* cur_scales;    // e4m3: [2][H]
  const char* mem_krot;       // this layer's ConvKV rotated keys [H][cap][D]
  const char* mem_v;
  int mem_cap;
  float scale;
  RopeDims rope;
  DevError* err;
};
cudaError_t launch_attn_simt(const AttnArgs& a, cudaStream_t s);

struct QrotArgs {
  const void* q;       // [T][H][D] bf16
  void* qrot;          // [S][H][T][D] bf16, or e4m3 codes when f8; when split:
                       // [S+1][H][T][D/2] bf16, dims 0..D/2-1 per slot and
                       // dims D/2..D-1 (no temporal pair) once, at slot S
  float* qscale;       // f8: [H][T] per-token scales
  const DevContext* ctx;
  int T, H, D, n_qrot;
  int f8;
  int split;           // bf16 with every temporal dim below D/2 (layout above)
  RopeDims rope;
  DevError* err;
};
cudaError_t launch_qrot(const QrotArgs& a, cudaStream_t s);

struct TcAttnArgs {
  CUtensorMap tm_q;    // rotated queries  [S*H][T][D] bf16 (e4m3 codes when kv_f8),
                       // or [(S+1)*H][T][D/2] bf16 when q_shared_z >= 0
  CUtensorMap tm_kv;   // pool pages       [frames*G*H][T][D] kv dtype (whole pool)
  CUtensorMap tm_cur;  // current pages    [2*H][T][D]
  CUtensorMap tm_mem;  // ConvKV rings     [L*3*H][cap][D] (or a dummy)
  const DevContext* ctx;
  const int* sched;           // work items per CTA (attn_tc_schedule for `grid`)
  int grid;                   // CTAs (attn_tc_schedule's return value)
  int n_pieces;               // pieces per head of a split query tile (0: none)
  float* part_o;              // pieces: [H][n_pieces][128][D] fp32, v_max * O unnormalised
  float2* part_ml;            // pieces: [H][n_pieces][128] (running max, sum)
  const float* frame_scales;  // e4m3: this layer's [n_frames][2][H]
  const float* cur_scales;    // e4m3: [2][H]
  const float* q_scales;      // e4m3: [H][T]
  int n_frames;               // frames per layer (bound of ctx->frame)
  int kv_f8;                  // 1: e4m3 K/V and queries, kind::f8f6f4
  int q_shared_z;             // >= 0: split query rows; the second half of head h's
                              // rows sits at map z = q_shared_z + h (one copy for all slots)
  uint64_t timeout_ns;        // limit of every wait in the kernel
  int stall;                  // failure injection: the MMA thread first waits on a
                              // barrier nothing completes (runs into timeout_ns)
  void* out;           // [T][H][D] bf16
  int T, H;
  int layer_frame0;    // first frame page row of this layer in tm_kv, in pages
  int G;
  int mem_row0;        // first row (in H-units) of this layer's rings in tm_mem
  float scale_log2;
  DevError* err;
};
cudaError_t launch_attn_tc(const TcAttnArgs& a, int num_sms, cudaStream_t s);
// Work items of the tensor-core attention: full units (two query tiles) and,
// when a head has an odd number of query tiles, n_pieces pieces per head of
// its last tile (one per context slot; n_pieces = the most slots a context
// has, attn_tc_pieces gives 0 when there is no odd tile).
int attn_tc_pieces(int T, int n_slots_max);
int attn_tc_items(int T, int H, int n_pieces);
size_t attn_tc_sched_ints(int T, int H, int n_pieces);   // bound of the table's size
// Deals the items to at most num_sms CTAs; returns the grid G and fills out
// with G + 1 offsets followed by each CTA's items.
int attn_tc_schedule(int T, int H, int n_pieces, int num_sms, int* out);
bool attn_tc_supported(int D, int kv_dtype);

// Combines the pieces of the split query tile into rows row0 .. T-1 of out.
struct MergeArgs {
  const DevContext* ctx;      // n_slots: pieces that hold results
  const float* part_o;
  const float2* part_ml;
  void* out;                  // [T][H][D] bf16
  int T, H, row0, n_pieces;
  DevError* err;
};
cudaError_t launch_attn_merge(const MergeArgs& a, cudaStream_t s);

}  // namespace la
