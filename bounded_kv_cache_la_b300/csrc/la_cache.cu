// Host state machine and C ABI of the bounded KV cache.
//
// The cache follows "LiveAnimate" (ai-feeds.com) 方法 for PR-Sink -- static
// sink (block 0 kept forever), dynamic sink (pose top-k), rolling window of
// the 3 most recent blocks, current block -- and "SoulX-LiveAct"
// (youleyou.com) 技术内核 for ConvKV -- exact window + current block, older
// blocks conv-compressed into a fixed FIFO memory with reset positions.
//
// Memory: everything lives in one caller-owned device pool, carved into
// regions (Layout).  K/V are stored per (layer, frame) in pages laid out
// [H][T][D]; a frame is the page group of one block.  The host tracks which
// block holds which frame, the window, the dynamic picks and the ConvKV ring;
// the per-block slot table is uploaded once per block and read by every
// attention launch of that block.
#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdio>
#include <cstring>
#include <deque>
#include <map>
#include <string>
#include <vector>

#include <nvtx3/nvToolsExt.h>

#include "la_internal.h"

using namespace la;

struct la_cache {
  la_cache_config cfg{};
  char* pool = nullptr;
  size_t pool_bytes = 0;
  Layout L{};
  const void* conv_w = nullptr;
  RopeDims rope{};
  int T = 0;
  int S_exact = 0;                  // largest number of exact slots
  int b = 0;                        // id of the block being generated
  bool selected = false;
  bool failed = false;
  std::string last_msg;
  la_context ctx{};
  DevContext dctx{}, dctx_final{};
  std::vector<int> frame_of;        // block -> frame (-1 none)
  std::vector<int> free_frames;
  std::deque<int> window;           // exact window blocks, oldest first
  std::vector<int> dyn;
  std::vector<int> pre;             // dynamic sink fetched ahead for block pre_for
  int pre_for = -1;
  std::vector<std::vector<char>> filled;   // [frame][layer] pages valid
  int cur_frame = -1;               // frame of the block being generated (set at select)
  std::vector<char> appended;
  std::vector<char> pages_written;  // [layer] the block's pages already hold its final K/V
  float query_kp[34] = {};
  int mem_n = 0, mem_head = 0;      // ConvKV ring state
  bool tc = false;
  bool q_split = false;          // split rotated-query layout (see QrotArgs)
  CUtensorMap tm_q{}, tm_kv{}, tm_cur{}, tm_mem{};
  std::vector<int> sched;           // tensor path: work items per CTA (uploaded)
  int attn_grid = 0;                // tensor path: CTAs of the attention launch
  int n_pieces = 0;                 // tensor path: pieces per head of a split query tile
  int num_sms = 148;
  std::vector<cudaEvent_t> prof_start, prof_stop;
  int inject_stall = 0;             // tensor-core launches still to stall (tests)
  int inject_bad_frame = 0;         // attention launches still to get a bad slot table (tests)
  DevContext dctx_inject{};         // host copy of that table (the upload reads it)
  size_t prof_next = 0;
};

namespace la {
static std::atomic<uint64_t> g_launches{0};
void count_launches(int n) { g_launches.fetch_add((uint64_t)n, std::memory_order_relaxed); }
}  // namespace la

namespace {

// NVTX range around a public call (shows the library's phases on a
// profiler timeline; costs nothing when no tool is attached).
struct Range {
  explicit Range(const char* name) { nvtxRangePushA(name); }
  ~Range() { nvtxRangePop(); }
};

constexpr size_t kAlign = 1024;
constexpr long long kMaxBlockTokens = 1 << 20;
size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

int elt_size(int dtype) { return dtype == LA_F32 ? 4 : dtype == LA_BF16 ? 2 : 1; }

bool is_prsink(const la_cache_config& c) { return c.policy == LA_POLICY_PR_SINK; }
// The kernels move Q/K/V/O rows and conv weights in 16-byte vectors.
bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }
bool is_external(const la_cache_config& c) { return c.history_mode == LA_HISTORY_EXTERNAL; }

la_status validate(const la_cache_config* c) {
  if (!c) return LA_ERR_INVALID_ARG;
  if (c->num_layers < 1 || c->num_heads < 1 || c->num_heads > 64) return LA_ERR_INVALID_ARG;
  if (c->head_dim != 64 && c->head_dim != 128) return LA_ERR_UNSUPPORTED;
  if (c->frames_per_block < 1 || c->grid_h < 1 || c->grid_w < 1) return LA_ERR_INVALID_ARG;
  // token indices are 32-bit in the kernels (divided by multiply-high below 2^31)
  if ((long long)c->frames_per_block * c->grid_h * c->grid_w > kMaxBlockTokens)
    return LA_ERR_UNSUPPORTED;
  if (c->rope_t < 0 || c->rope_h < 0 || c->rope_w < 0 || (c->rope_t | c->rope_h | c->rope_w) & 1 ||
      c->rope_t + c->rope_h + c->rope_w != c->head_dim)
    return LA_ERR_INVALID_ARG;
  if (!(c->rope_theta > 0.f)) return LA_ERR_INVALID_ARG;
  if (c->window < 1) return LA_ERR_INVALID_ARG;
  if (c->q_dtype != LA_F32 && c->q_dtype != LA_BF16) return LA_ERR_INVALID_ARG;
  if (c->kv_dtype != LA_F32 && c->kv_dtype != LA_BF16 && c->kv_dtype != LA_E4M3)
    return LA_ERR_INVALID_ARG;
  if (c->kv_dtype == LA_F32 && c->q_dtype != LA_F32) return LA_ERR_UNSUPPORTED;
  if (c->kv_dtype != LA_F32 && c->q_dtype != LA_BF16) return LA_ERR_UNSUPPORTED;
  if (!(c->softmax_scale > 0.f)) return LA_ERR_INVALID_ARG;
  if (c->attn_impl < LA_ATTN_AUTO || c->attn_impl > LA_ATTN_SIMT) return LA_ERR_INVALID_ARG;
  if (c->policy == LA_POLICY_PR_SINK) {
    if (c->static_sink < 0 || c->static_sink > 1) return LA_ERR_INVALID_ARG;
    if (c->dyn_topk < 0 || c->dyn_topk > LA_MAX_TOPK) return LA_ERR_INVALID_ARG;
    if (c->static_sink + c->dyn_topk + c->window + 1 > LA_MAX_SLOTS) return LA_ERR_INVALID_ARG;
    if (c->pose_dim != 34 || c->max_history < 1) return LA_ERR_INVALID_ARG;
    if (c->history_mode != LA_HISTORY_RESIDENT && c->history_mode != LA_HISTORY_EXTERNAL)
      return LA_ERR_INVALID_ARG;
  } else if (c->policy == LA_POLICY_CONVKV) {
    if (c->window + 1 > LA_MAX_SLOTS) return LA_ERR_INVALID_ARG;
    if (c->conv_kernel < 1 || c->conv_stride < 1 || c->mem_slots < 1) return LA_ERR_INVALID_ARG;
    int T = c->frames_per_block * c->grid_h * c->grid_w;
    if (T < c->conv_kernel) return LA_ERR_INVALID_ARG;
    int n_out = (T - c->conv_kernel) / c->conv_stride + 1;
    if (n_out > c->mem_slots) return LA_ERR_INVALID_ARG;
    if (c->kv_dtype != LA_BF16 || c->head_dim % 8) return LA_ERR_UNSUPPORTED;
  } else {
    return LA_ERR_INVALID_ARG;
  }
  return LA_OK;
}

int exact_slots(const la_cache_config& c) {
  return is_prsink(c) ? c.static_sink + c.dyn_topk + c.window + 1 : c.window + 1;
}

bool tc_eligible(const la_cache_config& c, const Layout& L) {
  if (c.attn_impl == LA_ATTN_SIMT) return false;
  // the e4m3 tensor path serves PR-Sink (the ConvKV memory is bf16)
  if (c.kv_dtype == LA_E4M3 && !is_prsink(c)) return false;
  return attn_tc_supported(c.head_dim, c.kv_dtype) && c.q_dtype == LA_BF16 &&
         L.page_stride == L.page_bytes;
}

void compute_layout(const la_cache_config& c, Layout& L) {
  const int H = c.num_heads, D = c.head_dim;
  const int T = c.frames_per_block * c.grid_h * c.grid_w;
  L.T = T;
  L.G = is_prsink(c) ? 2 : 3;
  if (is_prsink(c))
    // EXTERNAL: sink + window + current + dynamic sink, and as many again for
    // the next block's dynamic sink fetched ahead (la_prefetch_context)
    L.n_frames = is_external(c) ? c.static_sink + c.window + 1 + 2 * c.dyn_topk : c.max_history;
  else
    L.n_frames = c.window + 1;
  const int S = exact_slots(c);
  L.max_t = is_prsink(c) ? S * c.frames_per_block
                         : c.mem_slots + (c.window + 1) * c.frames_per_block;
  L.page_bytes = (size_t)H * T * D * elt_size(c.kv_dtype);
  L.page_stride = align_up(L.page_bytes, 256);
  L.n_qrot = S + (is_prsink(c) ? 0 : 1);
  const int hist = is_prsink(c) ? c.max_history : 1;

  size_t off = 0;
  auto take = [&](size_t bytes) {
    size_t o = off;
    off = align_up(off + bytes, kAlign);
    return o;
  };
  L.err = take(sizeof(DevError));
  L.ctx = take(sizeof(DevContext));
  L.ctx_final = take(sizeof(DevContext));
  L.ctx_inject = take(sizeof(DevContext));
  L.topk = take(sizeof(DevTopk));
  // e4m3 amax scratch, one [2][H] slice per frame plus one for the current
  // pages, so page writes to different frames may run on different streams
  L.amax = take(c.kv_dtype == LA_E4M3 ? sizeof(unsigned) * 2 * H * ((size_t)L.n_frames + 1)
                                      : sizeof(unsigned) * 2 * H);
  L.pose_tab = take(sizeof(float) * 36 * (size_t)hist);
  L.inv_norm = take(sizeof(float) * (size_t)hist);
  L.scores = take(sizeof(float) * (size_t)hist);
  L.rope_t = take(sizeof(float2) * (size_t)L.max_t * (c.rope_t / 2 > 0 ? c.rope_t / 2 : 1));
  L.rope_h = take(sizeof(float2) * (size_t)c.grid_h * (c.rope_h / 2 > 0 ? c.rope_h / 2 : 1));
  L.rope_w = take(sizeof(float2) * (size_t)c.grid_w * (c.rope_w / 2 > 0 ? c.rope_w / 2 : 1));
  L.scales = take(c.kv_dtype == LA_E4M3 ? sizeof(float) * c.num_layers * (size_t)L.n_frames * 2 * H : 0);
  L.cur_scales = take(sizeof(float) * 2 * H);
  L.frames = take((size_t)c.num_layers * L.n_frames * L.G * L.page_stride);
  L.cur_pages = take(2 * L.page_stride);
  const bool tc = tc_eligible(c, L);
  const bool f8 = c.kv_dtype == LA_E4M3;
  L.qrot = take(tc ? (size_t)L.n_qrot * H * T * D * (f8 ? 1 : 2) : 0);
  L.qscale = take(tc && f8 ? sizeof(float) * (size_t)H * T : 0);
  const int n_pieces = tc ? attn_tc_pieces(T, L.n_qrot) : 0;
  L.sched = take(tc ? sizeof(int) * attn_tc_sched_ints(T, H, n_pieces) : 0);
  L.part_o = take(sizeof(float) * (size_t)H * n_pieces * 128 * D);
  L.part_ml = take(sizeof(float2) * (size_t)H * n_pieces * 128);
  L.rope_t2 = take(tc && !f8 ? sizeof(float4) * (size_t)L.max_t * (c.rope_t / 2 > 0 ? c.rope_t / 2 : 1) : 0);
  L.mem = take(is_prsink(c) ? 0 : (size_t)c.num_layers * 3 * H * c.mem_slots * D * 2);
  L.total = off;
}

la_status cuda_status(la_cache* c, cudaError_t e, const char* what) {
  if (e == cudaSuccess) return LA_OK;
  c->failed = true;
  c->last_msg = std::string(what) + ": " + cudaGetErrorString(e);
  return LA_ERR_CUDA;
}

char* frame_page(la_cache* c, int layer, int frame, int which) {
  return c->pool + c->L.frames +
         (((size_t)layer * c->L.n_frames + frame) * c->L.G + which) * c->L.page_stride;
}
float* frame_scales(la_cache* c, int layer, int frame) {
  return reinterpret_cast<float*>(c->pool + c->L.scales) +
         ((size_t)layer * c->L.n_frames + frame) * 2 * c->cfg.num_heads;
}
char* mem_ring(la_cache* c, int layer, int which) {   // 0 raw K, 1 V, 2 rotated K
  const auto& g = c->cfg;
  return c->pool + c->L.mem +
         (((size_t)layer * 3 + which) * g.num_heads) * g.mem_slots * g.head_dim * 2;
}

int alloc_frame(la_cache* c) {
  if (c->free_frames.empty()) return -1;
  int f = c->free_frames.back();
  c->free_frames.pop_back();
  std::fill(c->filled[f].begin(), c->filled[f].end(), 0);
  return f;
}
void release_frame(la_cache* c, int block) {
  if (block < 0 || block >= (int)c->frame_of.size()) return;
  int f = c->frame_of[block];
  if (f < 0) return;
  c->frame_of[block] = -1;
  c->free_frames.push_back(f);
}

// Writes a block's K/V into frame pages (or the current pages when frame < 0).
la_status write_pages(la_cache* c, int layer, int frame, const void* k, const void* v,
                      bool with_raw, cudaStream_t s) {
  const auto& g = c->cfg;
  AppendArgs a{};
  a.k = k;
  a.v = v;
  if (frame >= 0) {
    a.k_dst = frame_page(c, layer, frame, 0);
    a.v_dst = frame_page(c, layer, frame, 1);
    a.kraw_dst = with_raw ? frame_page(c, layer, frame, 2) : nullptr;
    if (g.kv_dtype == LA_E4M3) {
      a.k_scale = frame_scales(c, layer, frame);
      a.v_scale = a.k_scale + g.num_heads;
    }
  } else {
    a.k_dst = c->pool + c->L.cur_pages;
    a.v_dst = c->pool + c->L.cur_pages + c->L.page_stride;
    a.kraw_dst = nullptr;
    a.k_scale = reinterpret_cast<float*>(c->pool + c->L.cur_scales);
    a.v_scale = a.k_scale + g.num_heads;
  }
  a.amax = reinterpret_cast<unsigned*>(c->pool + c->L.amax) +
           (g.kv_dtype == LA_E4M3 ? (size_t)(frame >= 0 ? frame : c->L.n_frames) * 2 * g.num_heads : 0);
  a.T = c->T;
  a.H = g.num_heads;
  a.D = g.head_dim;
  a.src_dtype = g.q_dtype;
  a.dst_dtype = g.kv_dtype;
  a.rope = c->rope;
  a.err = reinterpret_cast<DevError*>(c->pool + c->L.err);
  return cuda_status(c, launch_append(a, s), "append kernel");
}

void plan_slots(const la_cache_config& g, int b, const std::vector<int>& sink,
                const std::vector<int>& dyn, const std::vector<int>& win, int mem_n,
                la_context* out) {
  std::memset(out, 0, sizeof(*out));
  const int T = g.frames_per_block * g.grid_h * g.grid_w;
  out->block = b;
  out->mem_tokens = mem_n;
  int s = 0;
  auto push = [&](int id) {
    out->block_id[s] = id;
    out->t0[s] = mem_n + s * g.frames_per_block;
    ++s;
  };
  for (int id : sink) push(id);
  for (int id : dyn) push(id);
  for (int id : win) push(id);
  push(b);
  out->n_slots = s;
  out->kv_len = mem_n + s * T;
  out->n_dyn = (int)dyn.size();
  for (size_t i = 0; i < dyn.size(); ++i) out->dyn_ids[i] = dyn[i];
  out->topk_gap = INFINITY;
}

// Window contents when block b is generated (oldest first).
std::vector<int> window_blocks(const la_cache_config& g, int b) {
  std::vector<int> w;
  int first = std::max(0, b - g.window);
  for (int j = first; j < b; ++j) {
    if (is_prsink(g) && g.static_sink && j == 0) continue;
    w.push_back(j);
  }
  return w;
}

// 3D map [n_heads_total][rows_per_head][d] of 1- or 2-byte elements; a box
// is 128 rows x one 128-byte swizzled row span (64 bf16 or 128 e4m3).
bool encode_map(la_cache* c, CUtensorMap* m, void* base, int d, uint64_t rows_per_head,
                uint64_t n_heads_total, int elt) {
  typedef CUresult (*EncodeFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                               const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                               const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                               CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
  static EncodeFn fn = nullptr;
  if (!fn) {
    cudaDriverEntryPointQueryResult q;
    void* p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess || !p)
      return false;
    fn = reinterpret_cast<EncodeFn>(p);
  }
  cuuint64_t dims[3] = {(cuuint64_t)d, rows_per_head, n_heads_total};
  cuuint64_t strides[2] = {(cuuint64_t)d * elt, (cuuint64_t)d * elt * rows_per_head};
  cuuint32_t box[3] = {(cuuint32_t)(128 / elt), 128, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = fn(m, elt == 1 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3,
                  base, dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  (void)c;
  return r == CUDA_SUCCESS;
}

// Pose retrieval for block `blk` (query pose `kp`, written to table row
// blk): the top-k candidates (ids ascending, their scores) and the k-th /
// (k+1)-th score gap.  Synchronises `s` to read the picks.
la_status retrieve(la_cache* c, const float* kp, int blk, std::vector<int>& ids,
                   std::vector<float>& scores, float& gap, cudaStream_t s) {
  const auto& g = c->cfg;
  RetrievalArgs a{};
  std::memcpy(a.kp, kp, sizeof(a.kp));
  a.pose_row = blk;
  a.c0 = g.static_sink ? 1 : 0;
  a.c1 = std::max(a.c0, blk - g.window);
  a.k = g.dyn_topk;
  a.max_history = g.max_history;
  a.table = reinterpret_cast<float*>(c->pool + c->L.pose_tab);
  a.inv_norm = reinterpret_cast<float*>(c->pool + c->L.inv_norm);
  a.scores = reinterpret_cast<float*>(c->pool + c->L.scores);
  a.topk = reinterpret_cast<DevTopk*>(c->pool + c->L.topk);
  a.err = reinterpret_cast<DevError*>(c->pool + c->L.err);
  la_status st = cuda_status(c, launch_retrieval(a, s), "retrieval kernel");
  if (st != LA_OK) return st;
  DevError e{};
  DevTopk tk{};
  st = cuda_status(c, cudaMemcpyAsync(&tk, a.topk, sizeof(tk), cudaMemcpyDeviceToHost, s),
                   "read retrieval");
  if (st == LA_OK)
    st = cuda_status(c, cudaMemcpyAsync(&e, a.err, sizeof(DevError), cudaMemcpyDeviceToHost, s),
                     "read error word");
  if (st == LA_OK) st = cuda_status(c, cudaStreamSynchronize(s), "retrieval sync");
  if (st != LA_OK) return st;
  if (e.code != 0) {
    c->failed = true;
    return (la_status)e.code;
  }
  const int n = std::min(tk.n, g.dyn_topk);
  std::vector<std::pair<int, float>> picks;
  for (int i = 0; i < n; ++i) picks.push_back({tk.ids[i], tk.scores[i]});
  gap = INFINITY;
  if (tk.n > g.dyn_topk && g.dyn_topk > 0) gap = tk.scores[g.dyn_topk - 1] - tk.scores[g.dyn_topk];
  std::sort(picks.begin(), picks.end());
  ids.clear();
  scores.clear();
  for (auto& p : picks) {
    if (p.first < a.c0 || p.first >= a.c1) {
      c->failed = true;
      c->last_msg = "retrieval returned a non-candidate id";
      return LA_ERR_DEVICE;
    }
    ids.push_back(p.first);
    scores.push_back(p.second);
  }
  return LA_OK;
}

bool contains(const std::vector<int>& v, int x) { return std::find(v.begin(), v.end(), x) != v.end(); }

la_status check_usable(la_cache* c) {
  if (!c) return LA_ERR_INVALID_ARG;
  if (c->failed) return LA_ERR_STATE;
  return LA_OK;
}

}  // namespace

// ------------------------------------------------------------ checkpoint
// Host-state blob: magic, version, the config, then the block counter,
// fetch-ahead block, ConvKV ring position, the last query pose, and the
// frame table, free frames, dynamic sink, fetched-ahead picks and the
// per-frame / per-layer flags (each vector as a count and its elements).
namespace {
constexpr uint32_t kStateMagic = 0x5343414cu;   // "LACS"
constexpr uint32_t kStateVersion = 1;

struct Writer {
  std::vector<char> buf;
  template <class T> void put(const T& x) {
    const char* p = reinterpret_cast<const char*>(&x);
    buf.insert(buf.end(), p, p + sizeof(T));
  }
  template <class T> void put_vec(const std::vector<T>& v) {
    put<int64_t>((int64_t)v.size());
    for (const T& x : v) put(x);
  }
};
struct Reader {
  const char* p;
  size_t left;
  bool ok = true;
  template <class T> T get() {
    T x{};
    if (left < sizeof(T)) { ok = false; return x; }
    std::memcpy(&x, p, sizeof(T));
    p += sizeof(T);
    left -= sizeof(T);
    return x;
  }
  template <class T> std::vector<T> get_vec(int64_t max_n) {
    const int64_t n = get<int64_t>();
    std::vector<T> v;
    if (!ok || n < 0 || n > max_n) { ok = false; return v; }
    v.resize((size_t)n);
    for (auto& x : v) x = get<T>();
    return v;
  }
};

void write_state(const la_cache* c, Writer& w) {
  w.put(kStateMagic);
  w.put(kStateVersion);
  w.put(c->cfg);
  w.put<int32_t>(c->b);
  w.put<int32_t>(c->pre_for);
  w.put<int32_t>(c->mem_n);
  w.put<int32_t>(c->mem_head);
  for (float x : c->query_kp) w.put(x);
  w.put_vec(c->frame_of);
  w.put_vec(c->free_frames);
  w.put_vec(c->dyn);
  w.put_vec(c->pre);
  w.put_vec(std::vector<int>(c->window.begin(), c->window.end()));
  for (const auto& f : c->filled) w.put_vec(f);
}
}  // namespace

extern "C" {

const char* la_status_string(la_status s) {
  switch (s) {
    case LA_OK: return "ok";
    case LA_ERR_INVALID_ARG: return "invalid argument";
    case LA_ERR_OOM: return "pool too small";
    case LA_ERR_CUDA: return "CUDA runtime error";
    case LA_ERR_STATE: return "call out of order or earlier error";
    case LA_ERR_TIMEOUT: return "device wait timed out";
    case LA_ERR_UNSUPPORTED: return "unsupported configuration";
    case LA_ERR_DEVICE: return "kernel reported an out-of-range index";
  }
  return "unknown status";
}

size_t la_cache_required_bytes(const la_cache_config* cfg) {
  if (validate(cfg) != LA_OK) return 0;
  Layout L;
  compute_layout(*cfg, L);
  return L.total;
}

la_status la_context_plan(const la_cache_config* cfg, int block, const int32_t* dyn_ids,
                          int n_dyn, la_context* out) {
  la_status st = validate(cfg);
  if (st != LA_OK) return st;
  if (!out || block < 0 || n_dyn < 0 || (n_dyn > 0 && !dyn_ids)) return LA_ERR_INVALID_ARG;
  const auto& g = *cfg;
  std::vector<int> sink, dyn, win = window_blocks(g, block);
  int mem_n = 0;
  if (is_prsink(g)) {
    if (n_dyn > g.dyn_topk) return LA_ERR_INVALID_ARG;
    if (g.static_sink && block >= 1) sink.push_back(0);
    for (int i = 0; i < n_dyn; ++i) {
      int id = dyn_ids[i];
      bool cand = id >= (g.static_sink ? 1 : 0) && id < block - g.window;
      if (!cand || (i > 0 && id <= dyn_ids[i - 1])) return LA_ERR_INVALID_ARG;
      dyn.push_back(id);
    }
  } else {
    if (n_dyn) return LA_ERR_INVALID_ARG;
    const int T = g.frames_per_block * g.grid_h * g.grid_w;
    const long long per = (T - g.conv_kernel) / g.conv_stride + 1;
    const long long ev = std::max(0, block - g.window);
    mem_n = (int)std::min<long long>(g.mem_slots, per * ev);
  }
  plan_slots(g, block, sink, dyn, win, mem_n, out);
  return LA_OK;
}

int la_attention_schedule(int T, int H, int n_slots, int num_sms, int32_t* out, int cap) {
  if (T < 1 || T > kMaxBlockTokens || H < 1 || H > 64 || n_slots < 1 || n_slots > kMaxAttnSlots ||
      num_sms < 1 || !out)
    return -1;
  const int n_pieces = attn_tc_pieces(T, n_slots);
  std::vector<int> sched(attn_tc_sched_ints(T, H, n_pieces));
  const int G = attn_tc_schedule(T, H, n_pieces, num_sms, sched.data());
  const int n = G + 1 + sched[G];
  if (cap < n) return -1;
  for (int i = 0; i < n; ++i) out[i] = sched[i];
  return G;
}

// Builds the cache object over the caller's pool; init_pool: zero the
// control and ring regions and build the RoPE tables (a restored pool
// already holds them).
static la_status create_cache(const la_cache_config* cfg, void* dev_pool, size_t pool_bytes,
                              const void* conv_w, void* stream, bool init_pool, la_cache_t** out) {
  if (!out) return LA_ERR_INVALID_ARG;
  *out = nullptr;
  la_status st = validate(cfg);
  if (st != LA_OK) return st;
  if (!dev_pool || (reinterpret_cast<uintptr_t>(dev_pool) & 255)) return LA_ERR_INVALID_ARG;
  if (cfg->policy == LA_POLICY_CONVKV && (!conv_w || !aligned16(conv_w))) return LA_ERR_INVALID_ARG;
  Layout L;
  compute_layout(*cfg, L);
  if (pool_bytes < L.total) return LA_ERR_OOM;

  la_cache* c = new la_cache();
  c->cfg = *cfg;
  c->pool = static_cast<char*>(dev_pool);
  c->pool_bytes = pool_bytes;
  c->L = L;
  c->conv_w = conv_w;
  c->T = L.T;
  c->S_exact = exact_slots(*cfg);
  c->rope.dt = cfg->rope_t;
  c->rope.dh = cfg->rope_h;
  c->rope.dw = cfg->rope_w;
  c->rope.F = cfg->frames_per_block;
  c->rope.GH = cfg->grid_h;
  c->rope.GW = cfg->grid_w;
  c->rope.div_hw = make_fastdiv((uint32_t)(cfg->grid_h * cfg->grid_w));
  c->rope.div_w = make_fastdiv((uint32_t)cfg->grid_w);
  c->rope.max_t = L.max_t;
  c->rope.tab_t = reinterpret_cast<const float2*>(c->pool + L.rope_t);
  c->rope.tab_t2 = tc_eligible(*cfg, L) && cfg->kv_dtype != LA_E4M3
                       ? reinterpret_cast<const float4*>(c->pool + L.rope_t2)
                       : nullptr;
  c->rope.tab_h = reinterpret_cast<const float2*>(c->pool + L.rope_h);
  c->rope.tab_w = reinterpret_cast<const float2*>(c->pool + L.rope_w);
  const int hist = is_prsink(*cfg) ? cfg->max_history : 1;
  c->frame_of.assign(std::max(hist, 1024), -1);
  c->filled.assign(L.n_frames, std::vector<char>(cfg->num_layers, 0));
  if (!(is_prsink(*cfg) && !is_external(*cfg)))
    for (int f = L.n_frames - 1; f >= 0; --f) c->free_frames.push_back(f);
  c->appended.assign(cfg->num_layers, 0);
  c->pages_written.assign(cfg->num_layers, 0);

  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int dev = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&c->num_sms, cudaDevAttrMultiProcessorCount, dev);
  if (init_pool) st = cuda_status(c, cudaMemsetAsync(c->pool, 0, L.pose_tab, s), "pool init");
  if (st == LA_OK && init_pool)
    st = cuda_status(c,
                     launch_init_tables(reinterpret_cast<float2*>(c->pool + L.rope_t), L.max_t,
                                        cfg->rope_t, reinterpret_cast<float2*>(c->pool + L.rope_h),
                                        cfg->grid_h, cfg->rope_h,
                                        reinterpret_cast<float2*>(c->pool + L.rope_w), cfg->grid_w,
                                        cfg->rope_w, (double)cfg->rope_theta,
                                        const_cast<float4*>(c->rope.tab_t2), s),
                     "rope tables");
  if (st == LA_OK && init_pool && cfg->kv_dtype == LA_E4M3)
    st = cuda_status(c, cudaMemsetAsync(c->pool + L.scales, 0, L.frames - L.scales, s),
                     "scale init");
  // ConvKV rings start zeroed: attention reads whole tiles, so ring rows
  // past the valid count must hold finite values (they get weight 0).
  if (st == LA_OK && init_pool && !is_prsink(*cfg))
    st = cuda_status(c, cudaMemsetAsync(c->pool + L.mem, 0, L.total - L.mem, s), "memory init");
  c->tc = tc_eligible(*cfg, L);
  if (st == LA_OK && c->tc) {
    const int H = cfg->num_heads, D = cfg->head_dim;
    const int elt = cfg->kv_dtype == LA_E4M3 ? 1 : 2;
    // bf16 queries whose temporal pairs all sit in the first half of the head
    // dim: one rotated copy of the first half per slot, the second half once
    c->q_split = elt == 2 && cfg->rope_t <= D / 2;
    bool ok = (c->q_split ? encode_map(c, &c->tm_q, c->pool + L.qrot, D / 2, c->T,
                                       (uint64_t)(L.n_qrot + 1) * H, elt)
                          : encode_map(c, &c->tm_q, c->pool + L.qrot, D, c->T, (uint64_t)L.n_qrot * H, elt)) &&
              encode_map(c, &c->tm_kv, c->pool + L.frames, D, c->T,
                         (uint64_t)cfg->num_layers * L.n_frames * L.G * H, elt) &&
              encode_map(c, &c->tm_cur, c->pool + L.cur_pages, D, c->T, 2ull * H, elt);
    if (ok && !is_prsink(*cfg))
      ok = encode_map(c, &c->tm_mem, c->pool + L.mem, D, cfg->mem_slots,
                      (uint64_t)cfg->num_layers * 3 * H, 2);
    else if (ok)
      c->tm_mem = c->tm_cur;
    if (!ok) {
      c->failed = true;
      st = LA_ERR_CUDA;
      c->last_msg = "cuTensorMapEncodeTiled failed";
    }
    // the work-unit table depends on this device's SM count: built on every
    // create, a restored pool included
    if (st == LA_OK) {
      c->n_pieces = attn_tc_pieces(c->T, L.n_qrot);
      c->sched.assign(attn_tc_sched_ints(c->T, H, c->n_pieces), 0);
      c->attn_grid = attn_tc_schedule(c->T, H, c->n_pieces, c->num_sms, c->sched.data());
      const size_t n_ints = (size_t)c->attn_grid + 1 + c->sched[c->attn_grid];
      st = cuda_status(c, cudaMemcpyAsync(c->pool + L.sched, c->sched.data(), sizeof(int) * n_ints,
                                          cudaMemcpyHostToDevice, s),
                       "upload work-unit table");
    }
  }
  if (st != LA_OK) {
    delete c;
    return st;
  }
  *out = c;
  return LA_OK;
}

la_status la_cache_create(const la_cache_config* cfg, void* dev_pool, size_t pool_bytes,
                          const void* conv_w, void* stream, la_cache_t** out) {
  Range nvtx_range("la_cache_create");
  return create_cache(cfg, dev_pool, pool_bytes, conv_w, stream, true, out);
}


size_t la_cache_state_bytes(la_cache_t* c) {
  if (!c) return 0;
  Writer w;
  write_state(c, w);
  return w.buf.size();
}

la_status la_cache_save_state(la_cache_t* c, void* host_buf, size_t cap) {
  la_status st = check_usable(c);
  if (st != LA_OK) return st;
  if (!host_buf) return LA_ERR_INVALID_ARG;
  if (c->selected) return LA_ERR_STATE;           // only between blocks
  Writer w;
  write_state(c, w);
  if (cap < w.buf.size()) return LA_ERR_INVALID_ARG;
  std::memcpy(host_buf, w.buf.data(), w.buf.size());
  return LA_OK;
}

la_status la_cache_restore(const la_cache_config* cfg, void* dev_pool, size_t pool_bytes,
                           const void* conv_w, const void* state, size_t state_bytes, void* stream,
                           la_cache_t** out) {
  Range nvtx_range("la_cache_restore");
  if (!out) return LA_ERR_INVALID_ARG;
  *out = nullptr;
  if (!cfg || !state) return LA_ERR_INVALID_ARG;
  Reader r{static_cast<const char*>(state), state_bytes};
  const uint32_t magic = r.get<uint32_t>(), version = r.get<uint32_t>();
  const la_cache_config saved = r.get<la_cache_config>();
  if (!r.ok || magic != kStateMagic || version != kStateVersion ||
      std::memcmp(&saved, cfg, sizeof(saved)) != 0)
    return LA_ERR_INVALID_ARG;
  la_cache_t* c = nullptr;
  la_status st = create_cache(cfg, dev_pool, pool_bytes, conv_w, stream, false, &c);
  if (st != LA_OK) return st;
  const int32_t b = r.get<int32_t>(), pre_for = r.get<int32_t>();
  const int32_t mem_n = r.get<int32_t>(), mem_head = r.get<int32_t>();
  float kp[34];
  for (float& x : kp) x = r.get<float>();
  const int64_t max_ids = std::max<int64_t>(c->frame_of.size(), (int64_t)b * 2 + 2);
  auto frame_of = r.get_vec<int>(max_ids);
  auto free_frames = r.get_vec<int>(c->L.n_frames);
  auto dyn = r.get_vec<int>(LA_MAX_TOPK);
  auto pre = r.get_vec<int>(LA_MAX_TOPK);
  auto window = r.get_vec<int>(cfg->window);
  std::vector<std::vector<char>> filled(c->L.n_frames);
  for (auto& f : filled) {
    f = r.get_vec<char>(cfg->num_layers);
    if ((int)f.size() != cfg->num_layers) r.ok = false;
  }
  bool ok = r.ok && r.left == 0 && b >= 0 && mem_n >= 0 && mem_n <= cfg->mem_slots && mem_head >= 0 &&
            mem_head < std::max(cfg->mem_slots, 1) && (int64_t)frame_of.size() >= (int64_t)c->frame_of.size();
  for (int f : frame_of) ok = ok && f >= -1 && f < c->L.n_frames;
  for (int f : free_frames) ok = ok && f >= 0 && f < c->L.n_frames;
  // block ids index the frame table
  for (const auto* ids : {&dyn, &pre, &window})
    for (int id : *ids) ok = ok && id >= 0 && id < (int64_t)frame_of.size();
  if (!ok) {
    delete c;
    return LA_ERR_INVALID_ARG;
  }
  c->b = b;
  c->pre_for = pre_for;
  c->mem_n = mem_n;
  c->mem_head = mem_head;
  std::memcpy(c->query_kp, kp, sizeof(kp));
  c->frame_of = std::move(frame_of);
  c->free_frames = std::move(free_frames);
  c->dyn = std::move(dyn);
  c->pre = std::move(pre);
  c->window.assign(window.begin(), window.end());
  c->filled = std::move(filled);
  *out = c;
  return LA_OK;
}

la_status la_cache_destroy(la_cache_t* c) {
  if (!c) return LA_ERR_INVALID_ARG;
  delete c;
  return LA_OK;
}

la_status la_select_context(la_cache_t* c, const float* query_pose, la_context* out,
                            void* stream) {
  Range nvtx_range("la_select_context");
  la_status st = check_usable(c);
  if (st != LA_OK) return st;
  const auto& g = c->cfg;
  if (c->selected) return LA_ERR_STATE;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int b = c->b;
  std::vector<int> sink, dyn, win = window_blocks(g, b);
  std::vector<float> dyn_scores;
  float gap = INFINITY;
  for (int id : win)
    if (c->frame_of[id] < 0) return LA_ERR_STATE;   // window pages missing

  if (is_prsink(g)) {
    if (!query_pose) return LA_ERR_INVALID_ARG;
    if (b >= g.max_history) return LA_ERR_OOM;
    for (int i = 0; i < 34; ++i)
      if (!std::isfinite(query_pose[i])) return LA_ERR_INVALID_ARG;
    if (g.static_sink && b >= 1) {
      if (c->frame_of[0] < 0) return LA_ERR_STATE;
      sink.push_back(0);
    }
    std::memcpy(c->query_kp, query_pose, sizeof(c->query_kp));
    std::vector<float> scores;
    st = retrieve(c, query_pose, b, dyn, scores, gap, s);
    if (st != LA_OK) return st;
    dyn_scores = scores;
  }

  int mem_n = is_prsink(g) ? 0 : c->mem_n;
  la_context ctx;
  plan_slots(g, b, sink, dyn, win, mem_n, &ctx);
  ctx.topk_gap = gap;
  for (size_t i = 0; i < dyn_scores.size(); ++i) ctx.dyn_scores[i] = dyn_scores[i];

  // Dynamic-sink frames.  Blocks of the previous dynamic sink, or fetched
  // ahead for this block, that are not picked now (and are not the sink or
  // in the window) give their frames back.
  if (is_prsink(g) && is_external(g)) {
    std::vector<int> old = c->dyn;
    if (c->pre_for == b) old.insert(old.end(), c->pre.begin(), c->pre.end());
    for (int id : old)
      if (!contains(dyn, id) && !contains(win, id) && !(g.static_sink && id == 0))
        release_frame(c, id);
    c->pre.clear();
    c->pre_for = -1;
    for (size_t i = 0; i < dyn.size(); ++i) {
      int id = dyn[i];
      if (c->frame_of[id] < 0) {
        int f = alloc_frame(c);
        if (f < 0) {
          c->failed = true;
          c->last_msg = "no free frame for a dynamic-sink block";
          return LA_ERR_STATE;
        }
        c->frame_of[id] = f;
      }
      int f = c->frame_of[id];
      bool all = std::all_of(c->filled[f].begin(), c->filled[f].end(), [](char x) { return x; });
      ctx.need_fill[i] = all ? 0 : 1;
    }
  }
  c->dyn = dyn;

  // Device slot table.
  DevContext d{};
  int si = 0;
  if (mem_n > 0) {
    d.kind[si] = SLOT_MEMORY;
    d.frame[si] = -1;
    d.tokens[si] = mem_n;
    d.t0[si] = 0;               // memory keys carry their own positions
    ++si;
  }
  for (int e = 0; e < ctx.n_slots; ++e) {
    int id = ctx.block_id[e];
    if (id == b) {
      d.kind[si] = SLOT_CURRENT;
      d.frame[si] = -1;
    } else {
      d.kind[si] = SLOT_FRAME;
      d.frame[si] = c->frame_of[id];
    }
    d.tokens[si] = c->T;
    d.t0[si] = ctx.t0[e];
    ++si;
  }
  d.n_slots = si;
  d.kv_len = ctx.kv_len;
  d.t0_cur = ctx.t0[ctx.n_slots - 1];
  d.block = b;

  // The frame block b will occupy once committed.
  int fb;
  if (is_prsink(g) && !is_external(g)) {
    if (b >= c->L.n_frames) return LA_ERR_OOM;
    fb = b;
  } else {
    fb = alloc_frame(c);
    if (fb < 0) {
      c->failed = true;
      c->last_msg = "no free frame for the block being generated";
      return LA_ERR_STATE;
    }
  }
  // Same table with the current slot read from that frame: the last
  // denoising step of la_stream_step writes the block's pages there.
  DevContext dfin = d;
  dfin.kind[si - 1] = SLOT_FRAME;
  dfin.frame[si - 1] = fb;
  c->dctx = d;
  c->dctx_final = dfin;
  st = cuda_status(c, cudaMemcpyAsync(c->pool + c->L.ctx, &c->dctx, sizeof(d),
                                      cudaMemcpyHostToDevice, s),
                   "upload slot table");
  if (st == LA_OK)
    st = cuda_status(c, cudaMemcpyAsync(c->pool + c->L.ctx_final, &c->dctx_final, sizeof(d),
                                        cudaMemcpyHostToDevice, s),
                     "upload slot table");
  if (st != LA_OK) return st;
  c->ctx = ctx;
  c->selected = true;
  c->cur_frame = fb;
  std::fill(c->appended.begin(), c->appended.end(), 0);
  std::fill(c->pages_written.begin(), c->pages_written.end(), 0);
  if (out) *out = ctx;
  return LA_OK;
}

la_status la_fill_block(la_cache_t* c, int layer, int block_id, const void* k, const void* v,
                        void* stream) {
  Range nvtx_range("la_fill_block");
  la_status st = check_usable(c);
  if (st != LA_OK) return st;
  const auto& g = c->cfg;
  if (!is_prsink(g) || !is_external(g)) return LA_ERR_UNSUPPORTED;
  if (layer < 0 || layer >= g.num_layers || !k || !v || !aligned16(k) || !aligned16(v))
    return LA_ERR_INVALID_ARG;
  const bool cur = c->selected && contains(c->dyn, block_id);
  const bool ahead = c->pre_for >= c->b && contains(c->pre, block_id);
  if (!cur && !ahead) return c->selected || c->pre_for >= c->b ? LA_ERR_INVALID_ARG : LA_ERR_STATE;
  int f = c->frame_of[block_id];
  if (f < 0) return LA_ERR_STATE;
  st = write_pages(c, layer, f, k, v, false, static_cast<cudaStream_t>(stream));
  if (st == LA_OK) c->filled[f][layer] = 1;
  return st;
}

la_status la_prefetch_context(la_cache_t* c, const float* next_pose, la_context* out,
                              void* stream) {
  Range nvtx_range("la_prefetch_context");
  la_status st = check_usable(c);
  if (st != LA_OK) return st;
  const auto& g = c->cfg;
  if (!is_prsink(g) || !is_external(g)) return LA_ERR_UNSUPPORTED;
  if (!c->selected || c->pre_for == c->b + 1) return LA_ERR_STATE;
  if (!next_pose) return LA_ERR_INVALID_ARG;
  for (int i = 0; i < 34; ++i)
    if (!std::isfinite(next_pose[i])) return LA_ERR_INVALID_ARG;
  const int b1 = c->b + 1;
  if (b1 >= g.max_history) return LA_ERR_OOM;
  std::vector<int> ids;
  std::vector<float> scores;
  float gap = INFINITY;
  st = retrieve(c, next_pose, b1, ids, scores, gap, static_cast<cudaStream_t>(stream));
  if (st != LA_OK) return st;
  la_context ctx;
  std::vector<int> sink;
  if (g.static_sink) sink.push_back(0);
  plan_slots(g, b1, sink, ids, window_blocks(g, b1), 0, &ctx);
  ctx.topk_gap = gap;
  for (size_t i = 0; i < ids.size(); ++i) {
    const int id = ids[i];
    if (c->frame_of[id] < 0) {
      const int f = alloc_frame(c);
      if (f < 0) {
        c->failed = true;
        c->last_msg = "no free frame for a block fetched ahead";
        return LA_ERR_STATE;
      }
      c->frame_of[id] = f;
    }
    const int f = c->frame_of[id];
    ctx.dyn_scores[i] = scores[i];
    ctx.need_fill[i] = std::all_of(c->filled[f].begin(), c->filled[f].end(), [](char x) { return x; }) ? 0 : 1;
  }
  c->pre = ids;
  c->pre_for = b1;
  if (out) *out = ctx;
  return LA_OK;
}

la_status la_fill_window(la_cache_t* c, int layer, int block_id, const void* k, const void* v,
                         void* stream) {
  Range nvtx_range("la_fill_window");
  la_status st = check_usable(c);
  if (st != LA_OK) return st;
  const auto& g = c->cfg;
  if (!is_prsink(g) || !is_external(g)) return LA_ERR_UNSUPPORTED;
  if (layer < 0 || layer >= g.num_layers || !k || !v || !aligned16(k) || !aligned16(v))
    return LA_ERR_INVALID_ARG;
  std::vector<int> win = window_blocks(g, c->b);
  bool ok = std::find(win.begin(), win.end(), block_id) != win.end() ||
            (g.static_sink && block_id == 0 && c->b >= 1);
  if (!ok || block_id < 0 || c->frame_of[block_id] < 0) return LA_ERR_INVALID_ARG;
  int f = c->frame_of[block_id];
  st = write_pages(c, layer, f, k, v, false, static_cast<cudaStream_t>(stream));
  if (st == LA_OK) c->filled[f][layer] = 1;
  return st;
}

la_status la_refresh_sink(la_cache_t* c, int layer, const void* k, const void* v, void* stream) {
  Range nvtx_range("la_refresh_sink");
  la_status st = check_usable(c);
  if (st != LA_OK) return st;
  const auto& g = c->cfg;
  if (!is_prsink(g) || !g.static_sink) return LA_ERR_UNSUPPORTED;
  if (layer < 0 || layer >= g.num_layers || !k || !v || !aligned16(k) || !aligned16(v))
    return LA_ERR_INVALID_ARG;
  if (c->selected || c->b < 1 || c->frame_of[0] < 0) return LA_ERR_STATE;
  const int f = c->frame_of[0];
  st = write_pages(c, layer, f, k, v, false, static_cast<cudaStream_t>(stream));
  if (st == LA_OK) c->filled[f][layer] = 1;
  return st;
}

la_status la_cache_load_history(la_cache_t* c, const float* kps, int n, void* stream) {
  Range nvtx_range("la_cache_load_history");
  la_status st = check_usable(c);
  if (st != LA_OK) return st;
  const auto& g = c->cfg;
  if (!is_prsink(g) || !is_external(g)) return LA_ERR_UNSUPPORTED;
  if (c->b != 0 || c->selected) return LA_ERR_STATE;
  if (!kps || n < 1 || n >= g.max_history) return LA_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  for (size_t i = 0; i < (size_t)n * 34; ++i)
    if (!std::isfinite(kps[i])) return LA_ERR_INVALID_ARG;
  // raw keypoints into the first 34 floats of each table row, then one
  // kernel turns every row into its descriptor
  float* table = reinterpret_cast<float*>(c->pool + c->L.pose_tab);
  st = cuda_status(c, cudaMemcpy2DAsync(table, 36 * sizeof(float), kps, 34 * sizeof(float),
                                        34 * sizeof(float), n, cudaMemcpyHostToDevice, s),
                   "upload pose history");
  if (st == LA_OK)
    st = cuda_status(c, launch_pose_rows(table, reinterpret_cast<float*>(c->pool + c->L.inv_norm), n, s),
                     "pose history");
  if (st != LA_OK) return st;
  c->b = n;
  std::vector<int> need = window_blocks(g, n);
  if (g.static_sink) need.insert(need.begin(), 0);
  for (int id : need) {
    int f = alloc_frame(c);
    if (f < 0) return LA_ERR_STATE;
    c->frame_of[id] = f;
  }
  std::vector<int> win = window_blocks(g, n);
  c->window.assign(win.begin(), win.end());
  return LA_OK;
}

}  // extern "C"

namespace {

// One chunk attention.  final = the last denoising step of the block inside
// la_stream_step: k_cur / v_cur are then also the block's final K/V, so they
// are written straight into the block's own frame (the slot table whose
// current slot is that frame is used) and the layer's append skips its copy.
la_status chunk_attention(la_cache* c, int layer, const void* q, const void* k_cur,
                          const void* v_cur, void* out, cudaStream_t s, bool final) {
  la_status st = check_usable(c);
  if (st != LA_OK) return st;
  const auto& g = c->cfg;
  if (!c->selected) return LA_ERR_STATE;
  if (layer < 0 || layer >= g.num_layers || !q || !k_cur || !v_cur || !out || !aligned16(q) ||
      !aligned16(k_cur) || !aligned16(v_cur) || !aligned16(out))
    return LA_ERR_INVALID_ARG;
  if (final && c->appended[layer]) return LA_ERR_STATE;
  if (is_prsink(g) && is_external(g)) {
    for (int e = 0; e < c->ctx.n_slots - 1; ++e) {
      int f = c->frame_of[c->ctx.block_id[e]];
      if (f < 0 || !c->filled[f][layer]) return LA_ERR_STATE;
    }
  }
  if (final) {
    st = write_pages(c, layer, c->cur_frame, k_cur, v_cur, !is_prsink(g), s);
    if (st != LA_OK) return st;
    c->filled[c->cur_frame][layer] = 1;
    c->pages_written[layer] = 1;
  } else {
    st = write_pages(c, layer, -1, k_cur, v_cur, false, s);
    if (st != LA_OK) return st;
  }
  const DevContext* dctx =
      reinterpret_cast<const DevContext*>(c->pool + (final ? c->L.ctx_final : c->L.ctx));
  if (c->inject_bad_frame > 0) {
    // failure injection: the first slot names a frame past the pool's frames
    --c->inject_bad_frame;
    c->dctx_inject = final ? c->dctx_final : c->dctx;
    c->dctx_inject.kind[0] = SLOT_FRAME;
    c->dctx_inject.frame[0] = c->L.n_frames + 7;
    st = cuda_status(c, cudaMemcpyAsync(c->pool + c->L.ctx_inject, &c->dctx_inject, sizeof(DevContext),
                                        cudaMemcpyHostToDevice, s),
                     "upload injected slot table");
    if (st != LA_OK) return st;
    dctx = reinterpret_cast<const DevContext*>(c->pool + c->L.ctx_inject);
  }
  DevError* err = reinterpret_cast<DevError*>(c->pool + c->L.err);
  if (c->tc) {
    QrotArgs qa{};
    qa.q = q;
    qa.qrot = c->pool + c->L.qrot;
    qa.ctx = dctx;
    qa.T = c->T;
    qa.H = g.num_heads;
    qa.D = g.head_dim;
    qa.n_qrot = c->L.n_qrot;
    qa.f8 = g.kv_dtype == LA_E4M3;
    qa.split = c->q_split;
    qa.qscale = reinterpret_cast<float*>(c->pool + c->L.qscale);
    qa.rope = c->rope;
    qa.err = err;
    st = cuda_status(c, launch_qrot(qa, s), "query rotation kernel");
    if (st != LA_OK) return st;
    TcAttnArgs ta{};
    ta.tm_q = c->tm_q;
    ta.tm_kv = c->tm_kv;
    ta.tm_cur = c->tm_cur;
    ta.tm_mem = c->tm_mem;
    ta.ctx = dctx;
    ta.sched = reinterpret_cast<const int*>(c->pool + c->L.sched);
    ta.grid = c->attn_grid;
    ta.n_pieces = c->n_pieces;
    ta.part_o = reinterpret_cast<float*>(c->pool + c->L.part_o);
    ta.part_ml = reinterpret_cast<float2*>(c->pool + c->L.part_ml);
    ta.kv_f8 = g.kv_dtype == LA_E4M3;
    ta.q_shared_z = c->q_split ? c->L.n_qrot * g.num_heads : -1;
    ta.frame_scales = ta.kv_f8 ? frame_scales(c, layer, 0) : nullptr;
    ta.cur_scales = reinterpret_cast<const float*>(c->pool + c->L.cur_scales);
    ta.q_scales = reinterpret_cast<const float*>(c->pool + c->L.qscale);
    ta.n_frames = c->L.n_frames;
    ta.out = out;
    ta.T = c->T;
    ta.H = g.num_heads;
    ta.layer_frame0 = layer * c->L.n_frames * c->L.G;
    ta.G = c->L.G;
    ta.mem_row0 = layer * 3 * g.num_heads;
    ta.scale_log2 = g.softmax_scale * 1.4426950408889634f;
    ta.stall = c->inject_stall > 0;
    if (ta.stall) --c->inject_stall;
    ta.timeout_ns = ta.stall ? 100000000ull : 2000000000ull;   // 0.1 s injected, else 2 s
    ta.err = err;
    const bool prof = c->prof_next < c->prof_start.size();
    if (prof) cudaEventRecord(c->prof_start[c->prof_next], s);
    st = cuda_status(c, launch_attn_tc(ta, c->num_sms, s), "tensor-core attention");
    if (st == LA_OK && c->n_pieces > 0) {
      // the last query tile, split by slot: combine its pieces
      MergeArgs ma{};
      ma.ctx = dctx;
      ma.part_o = ta.part_o;
      ma.part_ml = ta.part_ml;
      ma.out = out;
      ma.T = c->T;
      ma.H = g.num_heads;
      ma.row0 = (c->T / 256) * 256;
      ma.n_pieces = c->n_pieces;
      ma.err = err;
      st = cuda_status(c, launch_attn_merge(ma, s), "attention merge");
    }
    if (prof) cudaEventRecord(c->prof_stop[c->prof_next++], s);
    return st;
  }
  AttnArgs a{};
  a.q = q;
  a.out = out;
  a.T = c->T;
  a.H = g.num_heads;
  a.D = g.head_dim;
  a.q_dtype = g.q_dtype;
  a.kv_dtype = g.kv_dtype;
  a.ctx = dctx;
  a.frames = frame_page(c, layer, 0, 0);
  a.page_stride = c->L.page_stride;
  a.G = c->L.G;
  a.n_frames = c->L.n_frames;
  a.cur_k = c->pool + c->L.cur_pages;
  a.cur_v = c->pool + c->L.cur_pages + c->L.page_stride;
  a.frame_scales = g.kv_dtype == LA_E4M3 ? frame_scales(c, layer, 0) : nullptr;
  a.cur_scales = reinterpret_cast<const float*>(c->pool + c->L.cur_scales);
  a.mem_krot = is_prsink(g) ? nullptr : mem_ring(c, layer, 2);
  a.mem_v = is_prsink(g) ? nullptr : mem_ring(c, layer, 1);
  a.mem_cap = g.mem_slots;
  a.scale = g.softmax_scale;
  a.rope = c->rope;
  a.err = err;
  const bool prof = c->prof_next < c->prof_start.size();
  if (prof) cudaEventRecord(c->prof_start[c->prof_next], s);
  st = cuda_status(c, launch_attn_simt(a, s), "simt attention");
  if (prof) cudaEventRecord(c->prof_stop[c->prof_next++], s);
  return st;
}

}  // namespace

extern "C" {

la_status la_chunk_attention(la_cache_t* c, int layer, const void* q, const void* k_cur,
                             const void* v_cur, void* out, void* stream) {
  Range nvtx_range("la_chunk_attention");
  return chunk_attention(c, layer, q, k_cur, v_cur, out, static_cast<cudaStream_t>(stream), false);
}

la_status la_cache_append_block(la_cache_t* c, int layer, const void* k, const void* v,
                                void* stream) {
  Range nvtx_range("la_cache_append_block");
  la_status st = check_usable(c);
  if (st != LA_OK) return st;
  const auto& g = c->cfg;
  if (!c->selected) return LA_ERR_STATE;
  if (layer < 0 || layer >= g.num_layers || !k || !v || !aligned16(k) || !aligned16(v))
    return LA_ERR_INVALID_ARG;
  if (c->appended[layer]) return LA_ERR_STATE;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int b = c->b;
  if (c->cur_frame < 0) return LA_ERR_STATE;
  const bool convkv = !is_prsink(g);
  if (!c->pages_written[layer]) {
    st = write_pages(c, layer, c->cur_frame, k, v, convkv, s);
    if (st != LA_OK) return st;
    c->filled[c->cur_frame][layer] = 1;
  }

  if (convkv && (int)c->window.size() == g.window) {
    // The oldest exact block leaves the window: compress it into the memory.
    const int e = c->window.front();
    const int fe = c->frame_of[e];
    const int n_out = (c->T - g.conv_kernel) / g.conv_stride + 1;
    ConvArgs a{};
    a.kraw = frame_page(c, layer, fe, 2);
    a.v = frame_page(c, layer, fe, 1);
    a.w = static_cast<const char*>(c->conv_w) +
          (size_t)layer * 2 * g.num_heads * g.head_dim * g.conv_kernel * 2;
    a.k_ring = mem_ring(c, layer, 0);
    a.v_ring = mem_ring(c, layer, 1);
    a.krot_ring = mem_ring(c, layer, 2);
    a.T = c->T;
    a.H = g.num_heads;
    a.D = g.head_dim;
    a.R = g.conv_kernel;
    a.stride = g.conv_stride;
    a.n_out = n_out;
    a.cap = g.mem_slots;
    a.write0 = (c->mem_head + c->mem_n) % g.mem_slots;
    const int total = c->mem_n + n_out;
    a.n_after = std::min(total, g.mem_slots);
    a.head_after = total > g.mem_slots ? (c->mem_head + (total - g.mem_slots)) % g.mem_slots
                                       : c->mem_head;
    a.rope = c->rope;
    a.err = reinterpret_cast<DevError*>(c->pool + c->L.err);
    st = cuda_status(c, launch_convkv(a, s), "convkv kernel");
    if (st != LA_OK) return st;
  }
  c->appended[layer] = 1;
  if (!std::all_of(c->appended.begin(), c->appended.end(), [](char x) { return x; }))
    return LA_OK;

  // Commit block b.
  if (b >= (int)c->frame_of.size()) c->frame_of.resize((size_t)b * 2 + 1, -1);
  c->frame_of[b] = c->cur_frame;
  if (is_prsink(g) && g.static_sink && b == 0) {
    // block 0 is the static sink: kept forever, never in the window
  } else {
    c->window.push_back(b);
    if ((int)c->window.size() > g.window) {
      const int e = c->window.front();
      c->window.pop_front();
      // EXTERNAL: a block fetched ahead for the next block keeps its frame
      const bool ahead = is_external(g) && c->pre_for == b + 1 && contains(c->pre, e);
      if (!(is_prsink(g) && !is_external(g)) && !ahead) release_frame(c, e);
      if (convkv) {
        const int n_out = (c->T - g.conv_kernel) / g.conv_stride + 1;
        const int total = c->mem_n + n_out;
        if (total > g.mem_slots) {
          c->mem_head = (c->mem_head + (total - g.mem_slots)) % g.mem_slots;
          c->mem_n = g.mem_slots;
        } else {
          c->mem_n = total;
        }
      }
    }
  }
  c->cur_frame = -1;
  c->selected = false;
  c->b = b + 1;
  return LA_OK;
}

la_status la_stream_step(la_cache_t* c, const float* pose, int n_steps, const void* const* q,
                         const void* const* k, const void* const* v, void* const* out,
                         la_fill_fn fill, void* user, void* stream) {
  Range nvtx_range("la_stream_step");
  la_status st = check_usable(c);
  if (st != LA_OK) return st;
  const int L = c->cfg.num_layers;
  if (n_steps < 1 || !q || !k || !v || !out) return LA_ERR_INVALID_ARG;
  la_context ctx;
  st = la_select_context(c, pose, &ctx, stream);
  if (st != LA_OK) return st;
  for (int i = 0; i < ctx.n_dyn; ++i) {
    if (!ctx.need_fill[i]) continue;
    if (!fill) return LA_ERR_STATE;
    for (int l = 0; l < L; ++l) {
      st = fill(c, l, ctx.dyn_ids[i], user, stream);
      if (st != LA_OK) return st;
    }
  }
  for (int sidx = 0; sidx < n_steps; ++sidx)
    for (int l = 0; l < L; ++l) {
      size_t i = (size_t)sidx * L + l;
      st = chunk_attention(c, l, q[i], k[i], v[i], out[i], static_cast<cudaStream_t>(stream),
                           sidx == n_steps - 1);
      if (st != LA_OK) return st;
    }
  for (int l = 0; l < L; ++l) {
    size_t i = (size_t)(n_steps - 1) * L + l;
    st = la_cache_append_block(c, l, k[i], v[i], stream);
    if (st != LA_OK) return st;
  }
  return LA_OK;
}

la_status la_get_error(la_cache_t* c, char* msg, size_t cap) {
  Range nvtx_range("la_get_error");
  if (!c) return LA_ERR_INVALID_ARG;
  DevError e{};
  cudaError_t ce = cudaDeviceSynchronize();
  if (ce == cudaSuccess)
    ce = cudaMemcpy(&e, c->pool + c->L.err, sizeof(e), cudaMemcpyDeviceToHost);
  std::string m;
  la_status st = LA_OK;
  if (ce != cudaSuccess) {
    m = std::string("CUDA: ") + cudaGetErrorString(ce);
    st = LA_ERR_CUDA;
    c->failed = true;
  } else if (e.code != 0) {
    char buf[160];
    std::snprintf(buf, sizeof(buf), "kernel %d reported %s (detail %d, %d)", e.kernel,
                  la_status_string((la_status)e.code), e.detail0, e.detail1);
    m = buf;
    st = (la_status)e.code;
    c->failed = true;
  } else if (c->failed) {
    m = c->last_msg.empty() ? "earlier error" : c->last_msg;
    st = LA_ERR_STATE;
  } else {
    m = "ok";
  }
  if (msg && cap) {
    std::strncpy(msg, m.c_str(), cap - 1);
    msg[cap - 1] = 0;
  }
  return st;
}

la_status la_debug_page(la_cache_t* c, int layer, int block_id, int which, void** page,
                        void** scales) {
  if (!c || !page || layer < 0 || layer >= c->cfg.num_layers || which < 0 || which >= c->L.G ||
      block_id < 0 || block_id >= (int)c->frame_of.size())
    return LA_ERR_INVALID_ARG;
  int f = c->frame_of[block_id];
  if (f < 0) return LA_ERR_INVALID_ARG;
  *page = frame_page(c, layer, f, which);
  if (scales)
    *scales = c->cfg.kv_dtype == LA_E4M3 && which < 2 ? frame_scales(c, layer, f) + which * c->cfg.num_heads
                                                      : nullptr;
  return LA_OK;
}

la_status la_set_profile_events(la_cache_t* c, void* const* starts, void* const* stops, int n) {
  if (!c || n < 0 || (n > 0 && (!starts || !stops))) return LA_ERR_INVALID_ARG;
  c->prof_start.assign(n, nullptr);
  c->prof_stop.assign(n, nullptr);
  for (int i = 0; i < n; ++i) {
    c->prof_start[i] = static_cast<cudaEvent_t>(starts[i]);
    c->prof_stop[i] = static_cast<cudaEvent_t>(stops[i]);
  }
  c->prof_next = 0;
  return LA_OK;
}

uint64_t la_launch_count(void) { return la::g_launches.load(std::memory_order_relaxed); }

la_status la_debug_inject(la_cache_t* c, int what, int count) {
  if (!c || count < 0) return LA_ERR_INVALID_ARG;
  if (what == LA_INJECT_BAD_FRAME) {
    c->inject_bad_frame = count;
    return LA_OK;
  }
  if (what != LA_INJECT_ATTN_STALL) return LA_ERR_INVALID_ARG;
  if (!c->tc) return LA_ERR_UNSUPPORTED;
  c->inject_stall = count;
  return LA_OK;
}

la_status la_debug_memory(la_cache_t* c, int layer, void** k_raw, void** v, void** k_rot,
                          int* n_tokens, int* oldest) {
  if (!c || is_prsink(c->cfg) || layer < 0 || layer >= c->cfg.num_layers) return LA_ERR_INVALID_ARG;
  if (k_raw) *k_raw = mem_ring(c, layer, 0);
  if (v) *v = mem_ring(c, layer, 1);
  if (k_rot) *k_rot = mem_ring(c, layer, 2);
  if (n_tokens) *n_tokens = c->mem_n;
  if (oldest) *oldest = c->mem_head;
  return LA_OK;
}

}  // extern "C"
