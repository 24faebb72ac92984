// Fused gather + 3D-RoPE + flash attention on the tcgen05 tensor cores.
//
// "LiveAnimate" (ai-feeds.com) 方法: the current block attends, with no mask,
// to its bounded context (static sink, pose-retrieved dynamic sink, window of
// 3 blocks, itself); ConvKV ("SoulX-LiveAct" 技术内核) adds a compressed
// memory whose positions restart at 0.  Per head:
//     O = softmax(scale * R(Q) R(K_ctx)^T) V_ctx.
//
// RoPE.  Keys sit in the pool turned by their within-block position; the
// per-slot temporal offset is moved to the query side (scores depend only on
// position differences), so a query-rotation pass writes one rotated copy of
// Q per slot (for bf16 only the first half of each row, which holds every
// temporal pair, plus one shared copy of the second half) and the attention
// kernel itself does no trigonometry.
//
// Gather.  K/V tiles are TMA-loaded straight from the slot's pool page (the
// slot table says which page), 128 keys x 64 dims per box, 128-byte swizzle;
// rows past a slot's end are zero-filled by TMA and masked to -inf.
//
// Work.  A full unit is (head, pair of 128-row query tiles) against the
// whole context.  When a head has an odd number of query tiles, its last
// tile is split by context slot into pieces (the tile against one slot);
// each piece leaves its unnormalised output, running max and sum, and a
// small merge kernel combines them.  Dealt whole, that tile ran without a
// partner tile to overlap with and took 0.87 of a full unit: two of them
// on one CTA made it the slowest by 0.74 units (at 37 query tiles per head
// on 148 SMs).  A table built on the host lists each CTA's items; they are
// dealt by list scheduling in groups of about one round of heads (the full
// units, then the pieces, of each group), so pieces run beside their head's
// full units, read its K/V from L2 with them, and fill the end.
//
// CTA = 12 warps, persistent:
//   warp 0       TMA producer (K ring, V ring, per-slot Q boxes, double-buffered)
//   warp 1       MMA issuer: S_i = Q_i K^T (smem x smem) into TMEM,
//                O_i += P_i V (P from TMEM, V from smem, MN-major)
//   warp 2       TMEM allocator
//   warps 4..7   softmax of query tile 0 (one thread per row)
//   warps 8..11  softmax of query tile 1
// TMEM columns: S0 | S1 | O0 | O1 (128 each); P_i overwrites S_i as bf16.
// Issue order PV0(j-1), QK0(j), PV1(j-1), QK1(j) lets each softmax run while
// the tensor core works on the other tile.
//
// Softmax.  Base-2 online softmax with a lazy rescale: the running max moves
// only when a row's max grows by more than 8 (a factor 256), then O and l are
// rescaled.  The row max is only taken on a unit's first key tile or when a
// row's tile sum exceeds 2^8 (below that no value can pass the bound); it is
// a tree of 3-input maxes.  Scale-and-subtract and
// the row sum use packed fp32x2 arithmetic; the exponentials run on the MUFU
// unit (ex2.approx).  P is rounded to bf16 (relative error 2^-9) before the
// PV product (e4m3 with e4m3 operands).
//
// Every wait is bounded (2 s, or the injected limit); on timeout the kernel
// latches LA_ERR_TIMEOUT, drains its in-flight copies and MMAs, frees TMEM
// and returns.
#include <algorithm>
#include <vector>

#include "dev_common.cuh"
#include "tc_ptx.cuh"

namespace la {

namespace {

using namespace ptx;

constexpr int kBM = 128;                 // query rows per tile
constexpr int kBN = 128;                 // keys per tile
constexpr int kD = 128;                  // head dim
constexpr int kKSt = 2, kVSt = 2;
constexpr int kThreads = 384;
constexpr int kCtlBytes = 1024;
// Register split: launched at 168 per thread (384 threads, 1 CTA per SM =
// 64512).  Control warpgroup 128 x 112 + two softmax warpgroups 2 x 128 x 192
// = 63488: no spills in either region (88 / 208 spilled in the control code
// and measured the same).
constexpr int kRegsCtl = 112;
constexpr int kRegsSoftmax = 192;
static_assert(128 * kRegsCtl + 256 * kRegsSoftmax <= kThreads * 168, "register split too large");

// Per element type of Q/K/V/P in the MMAs: bf16 (kind::f16) or e4m3
// (kind::f8f6f4).  A tile is 128 rows of 128 elements, held as 128-byte
// swizzled rows: two 64-element boxes for bf16, one 128-element box for e4m3.
template <bool F8>
struct Tile {
  static constexpr int kElt = F8 ? 1 : 2;
  static constexpr int kBytes = kBM * kD * kElt;          // 32 KB / 16 KB
  static constexpr int kBoxes = F8 ? 1 : 2;
  static constexpr int kBoxBytes = kBytes / kBoxes;       // 16 KB
  static constexpr int kBoxElems = 128 / kElt;            // elements per 128-byte row
  static constexpr int kMmaK = F8 ? 32 : 16;              // K of one MMA instruction
  static constexpr int kSteps = kD / kMmaK;               // MMAs per 128-deep product
  // Query region, in 16 KB boxes: the slot-dependent box of each of the two
  // tiles, double-buffered (boxes 0-3: buffer b, tile i at 2b + i); bf16
  // adds the second 64-dim box of each tile (boxes 4-5), which is the same
  // for every slot when the rotated queries are split.
  static constexpr int kQBoxes = F8 ? 4 : 6;
  static constexpr int kOffQ = 0;
  static constexpr int kOffK = kOffQ + kQBoxes * kBoxBytes;
  static constexpr int kOffV = kOffK + kKSt * kBytes;
  static constexpr int kOffCtl = kOffV + kVSt * kBytes;
  static constexpr int kSmem = kOffCtl + kCtlBytes + 1024; // + alignment slack
  static_assert(kSmem <= 227 * 1024, "over the per-block shared memory limit");
};
constexpr float kRescaleThreshold = 8.0f;                 // log2(256)

struct Ctl {
  uint64_t q0_full[2], q0_empty[2];   // slot-dependent query boxes, per buffer
  uint64_t q1_full, q1_empty;         // bf16: second query boxes (per unit when split)
  uint64_t k_full[kKSt], k_empty[kKSt];
  uint64_t v_full[kVSt], v_empty[kVSt];
  uint64_t s_full[2], p_ready[2], o_full[2];
  uint64_t mma_done;
  uint64_t never;                  // failure injection: nothing arrives here
  uint32_t tmem_base;
  int abort_flag;
  DevContext ctx;
};
static_assert(sizeof(Ctl) <= kCtlBytes, "control block too large");

struct Wait {
  volatile int* abort_flag;
  DevError* err;
  uint64_t timeout_ns;
  __device__ __forceinline__ bool operator()(const uint64_t& bar, uint32_t parity, int where) const {
    const uint32_t b = smem_u32(&bar);
    if (mbar_try_wait(b, parity)) return true;
    const uint64_t t0 = globaltimer();
    for (uint32_t it = 1;; ++it) {
      if (mbar_try_wait(b, parity)) return true;
      if ((it & 31) == 0) {
        if (*abort_flag) return false;
        if (globaltimer() - t0 > timeout_ns) {
          *abort_flag = 1;
          record_error(err, LA_ERR_TIMEOUT, KID_ATTN_TC, where, blockIdx.x);
          return false;
        }
      }
    }
  }
};

// Work items.  Full units h * n_full + p: query tiles 2p, 2p+1 of head h
// against the whole context.  When a head has an odd number of query tiles,
// its last tile is split by context slot instead: piece H * n_full + h * P + s
// is that tile against slot s only (P = pieces per head, the most slots a
// context can have; pieces past the context's slots are empty).  A piece
// leaves its unnormalised output, running max and sum in `part`, and
// attn_merge_kernel combines the pieces.  sched holds the items of each CTA:
// sched[c] .. sched[c + 1] index the entries after the G + 1 offsets.
struct Units {
  int H, n_full, n_pieces, n_full_total;
  int begin, end;                   // this CTA's entries
  const int* items;
  __device__ Units(int T, int H_, int n_pieces_, const int* sched) : H(H_), n_pieces(n_pieces_) {
    const int nt_q = (T + kBM - 1) / kBM;
    n_full = nt_q / 2;
    n_full_total = H * n_full;
    begin = __ldg(sched + blockIdx.x);
    end = __ldg(sched + blockIdx.x + 1);
    items = sched + gridDim.x + 1;
  }
  // false when the CTA has no i-th item
  __device__ __forceinline__ bool get(int i, int& h, int& row0, bool& piece, int& slot) const {
    if (begin + i >= end) return false;
    const int u = __ldg(items + begin + i);
    if (u < n_full_total) {
      h = u / n_full;
      row0 = (u - h * n_full) * 2 * kBM;
      piece = false;
      slot = -1;
    } else {
      const int p = u - n_full_total;
      h = p / n_pieces;
      slot = p - h * n_pieces;
      row0 = n_full * 2 * kBM;
      piece = true;
    }
    return true;
  }
};

// Tensor map and row of slot s's key (which = 0) or value (which = 1) pages.
__device__ __forceinline__ const CUtensorMap* kv_map(const TcAttnArgs& a, const DevContext& c, int s,
                                                     int which, int h, int& row) {
  const int kind = c.kind[s];
  if (kind == SLOT_FRAME) {
    row = (a.layer_frame0 + c.frame[s] * a.G + which) * a.H + h;
    return &a.tm_kv;
  }
  if (kind == SLOT_CURRENT) {
    row = which * a.H + h;
    return &a.tm_cur;
  }
  row = a.mem_row0 + (which == 0 ? 2 : 1) * a.H + h;     // rotated-key ring / value ring
  return &a.tm_mem;
}

// Scales of slot s for head h (e4m3 cache): key scale (which = 0) or value
// scale (which = 1) of the block the slot holds.
__device__ __forceinline__ float slot_scale(const TcAttnArgs& a, const DevContext& c, int s, int which,
                                            int h) {
  if (c.kind[s] == SLOT_FRAME) return a.frame_scales[((size_t)c.frame[s] * 2 + which) * a.H + h];
  return a.cur_scales[which * a.H + h];
}

template <bool F8>
__global__ void __launch_bounds__(kThreads, 1) attn_tc_kernel(const __grid_constant__ TcAttnArgs a) {
  using Tl = Tile<F8>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  Ctl& ctl = *reinterpret_cast<Ctl*>(smem + Tl::kOffCtl);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t sQ = smem_u32(smem + Tl::kOffQ), sK = smem_u32(smem + Tl::kOffK),
                 sV = smem_u32(smem + Tl::kOffV);

  if (tid == 0) {
    for (int i = 0; i < 2; ++i) {
      mbar_init(smem_u32(&ctl.q0_full[i]), 1);
      mbar_init(smem_u32(&ctl.q0_empty[i]), 1);
    }
    mbar_init(smem_u32(&ctl.q1_full), 1);
    mbar_init(smem_u32(&ctl.q1_empty), 1);
    for (int i = 0; i < kKSt; ++i) {
      mbar_init(smem_u32(&ctl.k_full[i]), 1);
      mbar_init(smem_u32(&ctl.k_empty[i]), 1);
    }
    for (int i = 0; i < kVSt; ++i) {
      mbar_init(smem_u32(&ctl.v_full[i]), 1);
      mbar_init(smem_u32(&ctl.v_empty[i]), 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(smem_u32(&ctl.s_full[i]), 1);
      mbar_init(smem_u32(&ctl.p_ready[i]), 128);
      mbar_init(smem_u32(&ctl.o_full[i]), 1);
    }
    mbar_init(smem_u32(&ctl.mma_done), 1);
    mbar_init(smem_u32(&ctl.never), 1);
    ctl.abort_flag = 0;
    ctl.ctx = *a.ctx;
    fence_barrier_init();
  }
  if (warp == 2) {
    tmem_alloc(smem_u32(&ctl.tmem_base), 512);
    tmem_relinquish();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tmap(&a.tm_q);
    prefetch_tmap(&a.tm_kv);
    prefetch_tmap(&a.tm_cur);
    prefetch_tmap(&a.tm_mem);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();

  const DevContext& cx = ctl.ctx;
  const int n_slots = cx.n_slots;
  bool bad = n_slots < 1 || n_slots > kMaxAttnSlots;
  for (int s = 0; !bad && s < n_slots; ++s) {
    const int k = cx.kind[s], tok = cx.tokens[s];
    bad = tok < 1 || k < SLOT_FRAME || k > SLOT_MEMORY ||
          (k == SLOT_FRAME && (cx.frame[s] < 0 || cx.frame[s] >= a.n_frames)) ||
          (k != SLOT_MEMORY && tok > a.T) || (F8 && k == SLOT_MEMORY);
  }
  const Wait wait{&ctl.abort_flag, a.err, a.timeout_ns};
  const uint64_t limit_ns = a.timeout_ns;
  const uint32_t tmem = ctl.tmem_base;
  const Units units(a.T, a.H, a.n_pieces, a.sched);
  if (bad && tid == 0) record_error(a.err, LA_ERR_DEVICE, KID_ATTN_TC, n_slots, -1);

  if (warp < 4) {
   setmaxnreg_dec<kRegsCtl>();
   if (bad) {
   } else if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      uint32_t kc = 0, vc = 0, qc = 0, q1c = 0;
      bool ok = true;
      const bool split = a.q_shared_z >= 0;
      for (int i = 0; ok; ++i) {
        int h, row0, slot;
        bool piece;
        if (!units.get(i, h, row0, piece, slot)) break;
        if (piece && slot >= n_slots) continue;     // past this context's slots
        const int n_qt = piece ? 1 : 2;
        const int s_begin = piece ? slot : 0, s_end = piece ? slot + 1 : n_slots;
        for (int s = s_begin; ok && s < s_end; ++s) {
          const int nt = (cx.tokens[s] + kBN - 1) / kBN;
          int krow, vrow;
          const CUtensorMap* km = kv_map(a, cx, s, 0, h, krow);
          const CUtensorMap* vm = kv_map(a, cx, s, 1, h, vrow);
          for (int kt = 0; ok && kt < nt; ++kt) {
            const int ks = kc % kKSt;
            if (!(ok = wait(ctl.k_empty[ks], ((kc / kKSt) & 1) ^ 1, 1))) break;
            mbar_arrive_expect_tx(smem_u32(&ctl.k_full[ks]), Tl::kBytes);
            for (int bx = 0; bx < Tl::kBoxes; ++bx)
              tma_load_3d(sK + ks * Tl::kBytes + bx * Tl::kBoxBytes, km, bx * Tl::kBoxElems, kt * kBN,
                          krow, smem_u32(&ctl.k_full[ks]));
            ++kc;
            if (kt == 0) {
              // slot s's own query box (dims 0-63 for bf16, the whole row for
              // e4m3) into the buffer the slot before last used: it loads while
              // the previous slot is still being computed
              const int qb = qc & 1;
              if (!(ok = wait(ctl.q0_empty[qb], ((qc >> 1) & 1) ^ 1, 2))) break;
              mbar_arrive_expect_tx(smem_u32(&ctl.q0_full[qb]), n_qt * Tl::kBoxBytes);
              for (int qi = 0; qi < n_qt; ++qi)
                tma_load_3d(sQ + (2 * qb + qi) * Tl::kBoxBytes, &a.tm_q, 0, row0 + qi * kBM, s * a.H + h,
                            smem_u32(&ctl.q0_full[qb]));
              ++qc;
              // bf16 dims 64-127: once per unit when split (the same rows for
              // every slot), else with every slot
              if (!F8 && (!split || s == s_begin)) {
                if (!(ok = wait(ctl.q1_empty, (q1c & 1) ^ 1, 4))) break;
                mbar_arrive_expect_tx(smem_u32(&ctl.q1_full), n_qt * Tl::kBoxBytes);
                for (int qi = 0; qi < n_qt; ++qi)
                  tma_load_3d(sQ + (4 + qi) * Tl::kBoxBytes, &a.tm_q, split ? 0 : Tl::kBoxElems,
                              row0 + qi * kBM, split ? a.q_shared_z + h : s * a.H + h,
                              smem_u32(&ctl.q1_full));
                ++q1c;
              }
            }
            const int vs = vc % kVSt;
            if (!(ok = wait(ctl.v_empty[vs], ((vc / kVSt) & 1) ^ 1, 3))) break;
            mbar_arrive_expect_tx(smem_u32(&ctl.v_full[vs]), Tl::kBytes);
            for (int bx = 0; bx < Tl::kBoxes; ++bx)
              tma_load_3d(sV + vs * Tl::kBytes + bx * Tl::kBoxBytes, vm, bx * Tl::kBoxElems, kt * kBN,
                          vrow, smem_u32(&ctl.v_full[vs]));
            ++vc;
          }
        }
      }
      // Drain: the last loads issued on each ring must have landed before exit.
      for (uint32_t i = (kc > kKSt ? kc - kKSt : 0); i < kc; ++i) {
        const uint32_t b = smem_u32(&ctl.k_full[i % kKSt]);
        const uint64_t t0 = globaltimer();
        while (!mbar_try_wait(b, (i / kKSt) & 1) && globaltimer() - t0 < limit_ns) {}
      }
      for (uint32_t i = (vc > kVSt ? vc - kVSt : 0); i < vc; ++i) {
        const uint32_t b = smem_u32(&ctl.v_full[i % kVSt]);
        const uint64_t t0 = globaltimer();
        while (!mbar_try_wait(b, (i / kVSt) & 1) && globaltimer() - t0 < limit_ns) {}
      }
      for (uint32_t i = (qc > 2 ? qc - 2 : 0); i < qc; ++i) {
        const uint32_t b = smem_u32(&ctl.q0_full[i & 1]);
        const uint64_t t0 = globaltimer();
        while (!mbar_try_wait(b, (i >> 1) & 1) && globaltimer() - t0 < limit_ns) {}
      }
      if (q1c > 0) {
        const uint32_t b = smem_u32(&ctl.q1_full);
        const uint64_t t0 = globaltimer();
        while (!mbar_try_wait(b, (q1c - 1) & 1) && globaltimer() - t0 < limit_ns) {}
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      const uint32_t idesc_qk = F8 ? idesc_e4m3(kBM, kBN, 0, 0) : idesc_bf16(kBM, kBN, 0, 0);
      const uint32_t idesc_pv = F8 ? idesc_e4m3(kBM, kD, 0, 1) : idesc_bf16(kBM, kD, 0, 1);
      uint32_t kc = 0, vc = 0, qc = 0, q1c = 0, pc0 = 0, pc1 = 0;
      bool ok = true;
      const bool split = a.q_shared_z >= 0;
      if (a.stall) ok = wait(ctl.never, 0, 31);     // injected: runs out, latches a timeout
      // Shared-memory descriptors are built once; a tile or K-step offset is
      // added to the 14-bit start-address field (addresses >> 4, all below
      // 256 KB, so the add never carries out of the field).  Few
      // instructions per MMA matter: this thread shares its sub-partition's
      // issue slots with two softmax warps.
      const uint64_t dq0 = sdesc(sQ, 16, 1024), dk0 = sdesc(sK, 16, 1024);
      const uint64_t dv0 = sdesc(sV, Tl::kBoxBytes, 1024);
      // S_i = Q_i K^T: both K-major; step kk covers 32 bytes of each 128-byte
      // row.  Query tile i's first box sits in buffer qb, its second (bf16)
      // in the per-tile box after the two buffers.
      auto issue_qk = [&](int i, int ks, int qb) {
        const uint64_t q0 = dq0 + ((uint32_t)((2 * qb + i) * Tl::kBoxBytes) >> 4);
        const uint64_t q1 = dq0 + ((uint32_t)((4 + i) * Tl::kBoxBytes) >> 4);
        const uint64_t k = dk0 + ((uint32_t)(ks * Tl::kBytes) >> 4);
#pragma unroll
        for (int kk = 0; kk < Tl::kSteps; ++kk) {
          const uint32_t in_box = ((kk * 32) % 128) >> 4;
          const uint64_t qd = (kk * 32 < 128 ? q0 : q1) + in_box;
          const uint32_t off = ((kk * 32 / 128) * Tl::kBoxBytes + (kk * 32) % 128) >> 4;
          if (F8)
            mma_ss_f8(tmem + i * 128, qd, k + off, idesc_qk, kk > 0);
          else
            mma_ss(tmem + i * 128, qd, k + off, idesc_qk, kk > 0);
        }
      };
      // O_i += P_i V: P from TMEM (8 columns per step), V MN-major (kMmaK key
      // rows of 128 bytes per step, 128-byte column chunks kBoxBytes apart).
      auto issue_pv = [&](int i, int vs, bool first) {
        const uint64_t v = dv0 + ((uint32_t)(vs * Tl::kBytes) >> 4);
#pragma unroll
        for (int kk = 0; kk < Tl::kSteps; ++kk) {
          const uint64_t bd = v + ((uint32_t)(kk * Tl::kMmaK * 128) >> 4);
          if (F8)
            mma_ts_f8(tmem + 256 + i * 128, tmem + i * 128 + kk * 8, bd, idesc_pv, !(first && kk == 0));
          else
            mma_ts(tmem + 256 + i * 128, tmem + i * 128 + kk * 8, bd, idesc_pv, !(first && kk == 0));
        }
      };
      for (int i = 0; ok; ++i) {
        int h, row0, slot;
        bool piece;
        if (!units.get(i, h, row0, piece, slot)) break;
        if (piece && slot >= n_slots) continue;      // past this context's slots
        const int s_begin = piece ? slot : 0, s_end = piece ? slot + 1 : n_slots;
        int j = 0;
        for (int s = s_begin; ok && s < s_end; ++s) {
          const int nt = (cx.tokens[s] + kBN - 1) / kBN;
          const int qb = qc & 1;                      // this slot's query buffer
          const bool q1_new = !F8 && (!split || s == s_begin);
          const bool q1_last = !F8 && (!split || s == s_end - 1);
          for (int kt = 0; ok && kt < nt; ++kt, ++j) {
            const int ks = kc % kKSt;
            if (!(ok = wait(ctl.k_full[ks], (kc / kKSt) & 1, 11))) break;
            tc_fence_after();
            const int vs = vc % kVSt;
            if (j > 0) {
              if (!(ok = wait(ctl.p_ready[0], pc0 & 1, 12))) break;
              if (!(ok = wait(ctl.v_full[vs], (vc / kVSt) & 1, 13))) break;
              tc_fence_after();
              issue_pv(0, vs, j == 1);
              ++pc0;
            }
            if (kt == 0) {
              if (!(ok = wait(ctl.q0_full[qb], (qc >> 1) & 1, 14))) break;
              if (q1_new && !(ok = wait(ctl.q1_full, q1c & 1, 19))) break;
              tc_fence_after();
            }
            issue_qk(0, ks, qb);
            tc_commit(smem_u32(&ctl.s_full[0]));
            if (j > 0) {
              if (!piece) {
                if (!(ok = wait(ctl.p_ready[1], pc1 & 1, 15))) break;
                tc_fence_after();
                issue_pv(1, vs, j == 1);
                ++pc1;
              }
              tc_commit(smem_u32(&ctl.v_empty[vs]));
              ++vc;
            }
            if (!piece) {
              issue_qk(1, ks, qb);
              tc_commit(smem_u32(&ctl.s_full[1]));
            }
            tc_commit(smem_u32(&ctl.k_empty[ks]));
            ++kc;
            if (kt == nt - 1) {                       // the slot's last QK: its query boxes are free
              tc_commit(smem_u32(&ctl.q0_empty[qb]));
              ++qc;
              if (q1_last) {
                tc_commit(smem_u32(&ctl.q1_empty));
                ++q1c;
              }
            }
          }
        }
        if (!ok) break;
        // last tile of the unit
        const int vs = vc % kVSt;
        if (!(ok = wait(ctl.p_ready[0], pc0 & 1, 16))) break;
        if (!(ok = wait(ctl.v_full[vs], (vc / kVSt) & 1, 17))) break;
        tc_fence_after();
        issue_pv(0, vs, j == 1);
        ++pc0;
        tc_commit(smem_u32(&ctl.o_full[0]));
        if (!piece) {
          if (!(ok = wait(ctl.p_ready[1], pc1 & 1, 18))) break;
          tc_fence_after();
          issue_pv(1, vs, j == 1);
          ++pc1;
          tc_commit(smem_u32(&ctl.o_full[1]));
        }
        tc_commit(smem_u32(&ctl.v_empty[vs]));
        ++vc;
      }
      // every MMA issued has completed before TMEM is released
      tc_commit(smem_u32(&ctl.mma_done));
      const uint64_t t0 = globaltimer();
      while (!mbar_try_wait(smem_u32(&ctl.mma_done), 0) && globaltimer() - t0 < limit_ns) {}
    }
   }
  } else {
   setmaxnreg_inc<kRegsSoftmax>();
   if (!bad) {
    // ------------------------------------------------------------ softmax
    const int qi = (warp - 4) >> 2;                // query tile of this warpgroup
    const int quad = warp & 3;                     // TMEM lane quadrant of this warp
    const int r = quad * 32 + lane;                // row within the tile
    const uint32_t lane_off = (uint32_t)(quad * 32) << 16;
    const uint32_t tS = tmem + lane_off + qi * 128;
    const uint32_t tO = tmem + lane_off + 256 + qi * 128;
    uint32_t sph = 0, oph = 0;
    bool ok = true;
    for (int i = 0; ok; ++i) {
      int h, row0, slot;
      bool piece;
      if (!units.get(i, h, row0, piece, slot)) break;
      if (piece && (qi == 1 || slot >= n_slots)) continue;   // one query tile; past the context
      const int s_begin = piece ? slot : 0, s_end = piece ? slot + 1 : n_slots;
      const int row = row0 + qi * kBM + r;
      // e4m3: true score = q_scale(row) * k_scale(slot) * S; P is stored as
      // p * v_scale(slot) / v_max so that O = v_max * sum(P V codes).
      float q_scale = 1.f, v_max = 1.f;
      if (F8) {
        if (row < a.T) q_scale = a.q_scales[(size_t)h * a.T + row];
        v_max = 0.f;
        for (int s = 0; s < n_slots; ++s) v_max = fmaxf(v_max, slot_scale(a, cx, s, 1, h));
        if (!(v_max > 0.f)) v_max = 1.f;
      }
      float m = -INFINITY, l = 0.f;
      int j = 0;
      for (int s = s_begin; ok && s < s_end; ++s) {
        const int tokens = cx.tokens[s];
        const int nt = (tokens + kBN - 1) / kBN;
        // e4m3: P is stored as p * r, r = v_scale(slot) / v_max <= 1, by
        // shifting the exponent by log2(r); the row sum divides r back out.
        float c = a.scale_log2, lr = 0.f, inv_r = 1.f;
        if (F8) {
          c *= q_scale * slot_scale(a, cx, s, 0, h);
          const float r_slot = slot_scale(a, cx, s, 1, h) / v_max;
          lr = __log2f(r_slot);
          inv_r = 1.f / r_slot;
        }
        for (int kt = 0; kt < nt; ++kt, ++j) {
          ok = __all_sync(0xffffffffu, wait(ctl.s_full[qi], sph & 1, 21 + qi));
          if (!ok) break;
          ++sph;
          tc_fence_after();
          float sv[kBN];
          const int valid = tokens - kt * kBN;
          auto load_s = [&]() {
#pragma unroll
            for (int cc = 0; cc < 4; ++cc) tmem_ld32(tS + cc * 32, reinterpret_cast<uint32_t*>(sv) + cc * 32);
            tmem_wait_ld();
            if (valid < kBN) {
#pragma unroll
              for (int cc = 0; cc < kBN; ++cc)
                if (cc >= valid) sv[cc] = -INFINITY;
            }
          };
          // sv <- 2^(sv c - m + lr) in place; returns this row's sum of those.
          auto exp_tile = [&]() {
            const float2 c2 = make_float2(c, c), nm2 = make_float2(lr - m, lr - m);
            float2 acc[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f),
                             make_float2(0.f, 0.f)};
#pragma unroll
            for (int e = 0; e < kBN / 2; ++e) {
              const float2 x = ffma2(make_float2(sv[2 * e], sv[2 * e + 1]), c2, nm2);
              float2 p;
              p.x = ex2(x.x);
              p.y = ex2(x.y);
              sv[2 * e] = p.x;
              sv[2 * e + 1] = p.y;
              acc[e & 3] = fadd2(acc[e & 3], p);
            }
            const float2 s01 = fadd2(fadd2(acc[0], acc[1]), fadd2(acc[2], acc[3]));
            return s01.x + s01.y;
          };
          load_s();
          // Against the running max m no stored value may exceed 2^8 (e4m3
          // tops out at 448).  A row sum of at most 2^8 proves that without a
          // row max, so the max is only taken on a unit's first tile or when
          // some row's sum goes over; then the lazy rescale below applies and
          // the tile is recomputed.
          float tsum;
          bool exact = j == 0;
          for (;;) {
            if (exact) {
              // row max: 8 independent 3-input max chains, then a tree
              float t8[8];
#pragma unroll
              for (int e = 0; e < 8; ++e) t8[e] = fmax3(sv[e], sv[e + 8], sv[e + 16]);
#pragma unroll
              for (int b = 24; b + 16 <= kBN; b += 16)
#pragma unroll
                for (int e = 0; e < 8; ++e) t8[e] = fmax3(t8[e], sv[b + e], sv[b + 8 + e]);
#pragma unroll
              for (int e = 0; e < 8; ++e) t8[e] = fmaxf(t8[e], sv[kBN - 8 + e]);
              float mx = fmaxf(fmax3(t8[0], t8[1], t8[2]), fmax3(fmax3(t8[3], t8[4], t8[5]), t8[6], t8[7]));
              mx *= c;
              if (__any_sync(0xffffffffu, mx > m + kRescaleThreshold)) {
                const float m_new = fmaxf(m, mx);
                const float alpha = ex2(m - m_new);
                if (j > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {
#pragma unroll 1
                  for (int cc = 0; cc < 4; ++cc) {
                    uint32_t o[32];
                    tmem_ld32(tO + cc * 32, o);
                    tmem_wait_ld();
#pragma unroll
                    for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
                    tmem_st32(tO + cc * 32, o);
                  }
                  tmem_wait_st();
                }
                l *= alpha;
                m = m_new;
              }
            }
            tsum = exp_tile();
            if (exact || !__any_sync(0xffffffffu, !(tsum <= 256.f))) break;
            exact = true;
            load_s();
          }
          l += tsum * inv_r;
          if (!F8) {
#pragma unroll
            for (int hf = 0; hf < 2; ++hf) {
              uint32_t pk[32];
#pragma unroll
              for (int e = 0; e < 32; ++e) pk[e] = cvt_bf16x2(sv[hf * 64 + 2 * e], sv[hf * 64 + 2 * e + 1]);
              tmem_st32(tS + hf * 32, pk);
            }
          } else {
            uint32_t pk[32];
#pragma unroll
            for (int e = 0; e < 32; ++e) pk[e] = cvt_e4m3x4(sv[4 * e], sv[4 * e + 1], sv[4 * e + 2], sv[4 * e + 3]);
            tmem_st32(tS, pk);
          }
          tmem_wait_st();
          tc_fence_before();
          mbar_arrive(smem_u32(&ctl.p_ready[qi]));
        }
      }
      if (!ok) break;
      ok = __all_sync(0xffffffffu, wait(ctl.o_full[qi], oph & 1, 23 + qi));
      if (!ok) break;
      ++oph;
      tc_fence_after();
      if (piece) {
        // a piece: v_max * O (unnormalised, fp32), the running max and sum
        const size_t pi = (size_t)h * a.n_pieces + slot;
        float* po = a.part_o + (pi * kBM + r) * kD;
#pragma unroll
        for (int cc = 0; cc < 4; ++cc) {
          uint32_t o[32];
          tmem_ld32(tO + cc * 32, o);
          tmem_wait_ld();
          float4* d4 = reinterpret_cast<float4*>(po + cc * 32);
#pragma unroll
          for (int e = 0; e < 8; ++e)
            d4[e] = make_float4(__uint_as_float(o[4 * e]) * v_max, __uint_as_float(o[4 * e + 1]) * v_max,
                                __uint_as_float(o[4 * e + 2]) * v_max, __uint_as_float(o[4 * e + 3]) * v_max);
        }
        a.part_ml[pi * kBM + r] = make_float2(m, l);
        tc_fence_before();
        continue;
      }
      const float inv_l = v_max / l;
      uint16_t* dst = reinterpret_cast<uint16_t*>(a.out) + ((size_t)row * a.H + h) * kD;
#pragma unroll
      for (int cc = 0; cc < 4; ++cc) {
        uint32_t o[32];
        tmem_ld32(tO + cc * 32, o);
        tmem_wait_ld();
        uint32_t pk[16];
#pragma unroll
        for (int e = 0; e < 16; ++e)
          pk[e] = cvt_bf16x2(__uint_as_float(o[2 * e]) * inv_l, __uint_as_float(o[2 * e + 1]) * inv_l);
        if (row < a.T) {
          uint4* d4 = reinterpret_cast<uint4*>(dst + cc * 32);
#pragma unroll
          for (int e = 0; e < 4; ++e) d4[e] = make_uint4(pk[4 * e], pk[4 * e + 1], pk[4 * e + 2], pk[4 * e + 3]);
        }
      }
      tc_fence_before();
    }
   }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 2) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

}  // namespace

bool attn_tc_supported(int D, int kv_dtype) {
  return D == kD && (kv_dtype == LA_BF16 || kv_dtype == LA_E4M3);
}

int attn_tc_pieces(int T, int n_slots_max) { return ((T + kBM - 1) / kBM) & 1 ? n_slots_max : 0; }

int attn_tc_items(int T, int H, int n_pieces) {
  const int nt = (T + kBM - 1) / kBM;
  return H * (nt / 2) + ((nt & 1) ? H * n_pieces : 0);
}

size_t attn_tc_sched_ints(int T, int H, int n_pieces) { return 2 * (size_t)attn_tc_items(T, H, n_pieces) + 1; }

// List scheduling.  Items go, in order, to the CTA that is free first (by
// estimated time: a full unit 1, a piece 0.78 / P + 0.02 -- timestamps at
// 37 query tiles per head gave 0.129 of a full unit for each of 7 pieces
// and 0.106 for each of 9).  The order takes heads in
// groups of about one round (G / (n_full + 1/2) heads): a group's full units,
// then its pieces, so the pieces run beside their head's full units and read
// its K/V from L2 with them, and the short pieces fill the time the full
// units leave at the end.  Returns the grid G; out receives G + 1 offsets,
// then the items of CTA 0, CTA 1, ...
int attn_tc_schedule(int T, int H, int n_pieces, int num_sms, int* out) {
  const int nt = (T + kBM - 1) / kBM, n_full = nt / 2;
  const int P = (nt & 1) ? n_pieces : 0;
  const int n_items = attn_tc_items(T, H, n_pieces);
  const int G = n_items < num_sms ? n_items : num_sms;
  const int per_round = std::max(1, (int)(2.0 * G / (2 * n_full + 1) + 0.5));
  const double t_full = 1.0, t_piece = P > 0 ? 0.78 / P + 0.02 : 0.0;
  std::vector<std::vector<int>> list(G);
  std::vector<std::pair<double, int>> heap;
  for (int c = G - 1; c >= 0; --c) heap.emplace_back(0.0, c);
  auto cmp = [](const std::pair<double, int>& x, const std::pair<double, int>& y) {
    return x.first > y.first || (x.first == y.first && x.second > y.second);
  };
  std::make_heap(heap.begin(), heap.end(), cmp);
  auto deal = [&](int item, double t) {
    std::pop_heap(heap.begin(), heap.end(), cmp);
    auto& top = heap.back();
    list[top.second].push_back(item);
    top.first += t;
    std::push_heap(heap.begin(), heap.end(), cmp);
  };
  for (int h0 = 0; h0 < H; h0 += per_round) {
    const int h1 = std::min(H, h0 + per_round);
    for (int h = h0; h < h1; ++h)
      for (int p = 0; p < n_full; ++p) deal(h * n_full + p, t_full);
    for (int h = h0; h < h1; ++h)
      for (int sl = 0; sl < P; ++sl) deal(H * n_full + h * P + sl, t_piece);
  }
  int k = 0;
  for (int c = 0; c < G; ++c) {
    out[c] = k;
    for (int u : list[c]) out[G + 1 + k++] = u;
  }
  out[G] = k;
  return G;
}

// Merge of a split query tile: for each of its rows and head, the pieces'
// outputs O_s (times v_max), running maxima m_s and sums l_s combine as
//   O = sum_s 2^(m_s - M) O_s / sum_s 2^(m_s - M) l_s,  M = max_s m_s.
// One warp per row, 4 dims per lane.
__global__ void __launch_bounds__(128) attn_merge_kernel(const MergeArgs a) {
  const int r = blockIdx.x * 4 + (threadIdx.x >> 5);          // row within the tile
  const int h = blockIdx.y, lane = threadIdx.x & 31;
  const int row = a.row0 + r;
  if (row >= a.T) return;
  const int n = a.ctx->n_slots;
  if (n < 1 || n > a.n_pieces) {
    if (lane == 0 && r == 0 && h == 0) record_error(a.err, LA_ERR_DEVICE, KID_ATTN_TC, n, a.n_pieces);
    return;
  }
  const size_t base = (size_t)h * a.n_pieces;
  float M = -INFINITY;
  for (int sl = 0; sl < n; ++sl) M = fmaxf(M, a.part_ml[(base + sl) * kBM + r].x);
  float den = 0.f;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int sl = 0; sl < n; ++sl) {
    const float2 ml = a.part_ml[(base + sl) * kBM + r];
    const float w = exp2f(ml.x - M);
    den += w * ml.y;
    const float4 o = reinterpret_cast<const float4*>(a.part_o + ((base + sl) * kBM + r) * kD)[lane];
    acc.x += w * o.x;
    acc.y += w * o.y;
    acc.z += w * o.z;
    acc.w += w * o.w;
  }
  const float inv = 1.f / den;
  uint16_t* dst = reinterpret_cast<uint16_t*>(a.out) + ((size_t)row * a.H + h) * kD + lane * 4;
  *reinterpret_cast<uint2*>(dst) = make_uint2(cvt_bf16x2(acc.x * inv, acc.y * inv), cvt_bf16x2(acc.z * inv, acc.w * inv));
}

cudaError_t launch_attn_merge(const MergeArgs& a, cudaStream_t s) {
  if (a.n_pieces < 1 || a.T < 1 || a.H < 1 || a.H > 65535 || a.row0 >= a.T) return cudaErrorInvalidValue;
  const int rows = std::min(kBM, a.T - a.row0);
  attn_merge_kernel<<<dim3((rows + 3) / 4, a.H), 128, 0, s>>>(a);
  count_launches(1);
  return cudaGetLastError();
}

template <bool F8>
static cudaError_t launch_attn_tc_t(const TcAttnArgs& a, int num_sms, cudaStream_t s) {
  // the shared-memory opt-in is a per-device function attribute
  static bool configured[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!configured[dev]) {
    e = cudaFuncSetAttribute(attn_tc_kernel<F8>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             Tile<F8>::kSmem);
    if (e != cudaSuccess) return e;
    configured[dev] = true;
  }
  (void)num_sms;
  attn_tc_kernel<F8><<<a.grid, kThreads, Tile<F8>::kSmem, s>>>(a);
  count_launches(1);
  return cudaGetLastError();
}

cudaError_t launch_attn_tc(const TcAttnArgs& a, int num_sms, cudaStream_t s) {
  if (a.kv_f8 && a.q_shared_z >= 0) return cudaErrorInvalidValue;   // split rows are bf16 only
  return a.kv_f8 ? launch_attn_tc_t<true>(a, num_sms, s) : launch_attn_tc_t<false>(a, num_sms, s);
}

}  // namespace la
