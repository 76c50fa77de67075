// Chunked append-prefill attention on a reused prefix.
//
// What it computes (definition): new token i of sequence b sits at absolute
// position p0 + i (p0 = prefix length) and, for each query head h, attends
// the keys [lo, p0 + i] of its own sequence, where lo = 0 for a global layer
// or max(0, p0 + i + 1 - window) for a local one: softmax of
// softmax_scale * <q, s_k[t] * k_code[t]> and the weighted sum of
// s_v[t] * v_code[t].  The prefix keys are read back from the int8 cache, not
// recomputed (prefix caching, Red Hat page "3. Cache de prefixo"; cross-turn
// cache, "Character.AI: inference optimization" section 04), and the chunk's
// own keys were appended to the same pages before this call.
//
// How:
//  1. dequant pass: the keys the chunk can see are copied into a contiguous
//     scratch copy: K codes as bf16 [B][KT][128] (exact), the per-key K scale
//     times softmax_scale * log2(e) as fp32 [B][KT], and V already multiplied by
//     its per-key scale, rounded once to fp16 [B][KT][128] (relative error at
//     most 2^-11, the same as the rounding of P).
//  2. attention: a persistent kernel whose work items are pairs of 128-row
//     q-tiles of one sequence, a row being one (new token, head) pair.  128-key
//     tiles of K and V arrive by TMA tensor loads (cp.async.bulk.tensor)
//     straight into the canonical no-swizzle tcgen05 operand layout; S = Q K^T
//     runs as tcgen05.mma kind::f16 (bf16, M = N = 128, K = 128) into tensor
//     memory; the online softmax (one thread per row, one warpgroup per q-tile
//     so each works while the tensor core runs the other's MMAs) forms
//     logit - reference with one FFMA per key (per-key K scale), applies the
//     causal/window mask on boundary tiles only, raises the reference lazily
//     (when a logit exceeds it by 2^8), and writes P (fp16) back into tensor
//     memory, where it is the A operand of O += P V' (V' from shared memory,
//     MN-major).
#include <cuda_fp16.h>

#include "common.cuh"
#include "tma.cuh"
#include "ptx.cuh"

namespace cai {
namespace {

constexpr int kRows = 128;                 // query rows per q-tile (MMA M)
constexpr int kQT = 2;                     // q-tiles per CTA sharing each K/V tile
constexpr int kKeys = 128;                 // keys per tile (MMA N of S, K of PV)
constexpr int kTileBytes = kKeys * kHeadDim * 2;  // 32 KB of 16-bit values
constexpr int kStages = 2;
constexpr int kOffQ = 0;                                     // Q[kQT]
// K tiles and V tiles (with the tile's K scales) have separate two-slot rings: a K
// slot is free as soon as both q-tiles' S = Q K^T have run, so the next K tile loads
// while the softmax of this one runs; a V slot (and its scales, which the softmax
// reads) is free after both PVs.
constexpr int kOffK = kOffQ + kQT * kRows * kHeadDim * 2;   // K[kStages]
constexpr int kVSlotBytes = kTileBytes + kKeys * 4;          // V (scaled), K scales
constexpr int kOffV = kOffK + kStages * kTileBytes;          // V[kStages]
constexpr int kOffBars = kOffV + kStages * kVSlotBytes;
constexpr int kNumBars = 4 * kStages + 6 * kQT + 1;  // ... and the MMA issuer's last commit
constexpr int kOffMisc = kOffBars + 8 * kNumBars;
constexpr int kSmemBytes = kOffMisc + 24 + 1024;  // tmem slot, wait state (+8); alignment slack
// Warpgroup 0: K/V producer (warp 0), MMA issuer (warp 1), two spare warps;
// warpgroups 1 and 2: the softmax of q-tile 0 and q-tile 1.  The block is
// launched with 168 registers per thread (384 threads; 3 warps x 32 x 168 =
// 16128 of a sub-partition's 16384), then warpgroup 0 shrinks to 72 and the
// softmax groups grow to 216: 128 * (72 + 216 + 216) = 64512 = 384 * 168, so
// the growth is covered exactly by what warpgroup 0 gives back.  The host
// checks the launch register count before the first launch.
constexpr int kThreads = 384;
constexpr int kRegsCtl = 72, kRegsSoft = 216;
constexpr int kRegsLaunch = 168;
static_assert(kRegsCtl * 128 + kRegsSoft * 256 <= kRegsLaunch * kThreads, "register split");
constexpr uint32_t kTmemCols = 512;        // per q-tile: S (128 columns, P over its first 64) + O (128)
constexpr float kRescaleThreshold = 8.0f;

struct PrefillParams {
  const uint8_t* pages;
  int32_t num_pages, page_size, max_pages;
  const int32_t* table;
  const int32_t* prefix_len;
  const uint16_t* q;      // bf16 [rows of new tokens][Hq][128], sequence b's rows from q_row0(b)
  const int32_t* q_off;   // [B + 1] packed new-token offsets, or null: sequence b has n_new rows at b * n_new
  int32_t batch, n_new, total_new, num_heads, log2_heads, window, kt_rows, pairs;  // n_new: the most per sequence
  float scale_log2;
  // Work items: items [0, full_items) are whole pairs of q-tiles; the pairs after them
  // (the last, partial wave of a persistent grid) are cut into `pieces` key ranges each,
  // item full_items + t being piece t % pieces of pair full_items + t / pieces.  A piece
  // writes its normalised partial output and log2-sum-exp to piece_o / piece_lse
  // ([t][256 rows][128] and [t][256]); combine_pieces_kernel merges them.
  int32_t full_items, pieces, num_items;
  uint64_t wait_ns;  // limit of every bounded wait inside the kernel
  int32_t drop_stage;  // fault injection: K tile each CTA skips (-1: none)
  int32_t skip_single;  // see PrefillLaunch
  float* piece_o;
  float* piece_lse;
  uint16_t* kb;  // scratch bf16 [B][KT][128]
  uint16_t* vh;  // scratch fp16 [B][KT][128]: V codes times the V scale
  float* ks;     // scratch [B][KT]: K scale * softmax scale * log2(e)
  float* out;
  float* lse_out;
  int32_t* err;
};

// New tokens of sequence b: rows [r0, r0 + n) of q / out, or n = -1 when its offsets
// are out of order or outside [0, total_new] (nothing of it is read or written).
struct SeqRows {
  int64_t r0;
  int n;
};

__device__ __forceinline__ SeqRows seq_rows(const PrefillParams& p, int b) {
  SeqRows s;
  if (!p.q_off) {
    s.r0 = (int64_t)b * p.n_new;
    s.n = p.n_new;
    return s;
  }
  const int32_t a = p.q_off[b], e = p.q_off[b + 1];
  s.r0 = a;
  s.n = (a >= 0 && a <= e && e <= p.total_new && e - a <= p.n_new) ? e - a : -1;
  if (p.skip_single && s.n == 1) s.n = 0;  // decoded by the decode kernel in the same call
  return s;
}

__device__ __forceinline__ bool seq_ok(const PrefillParams& p, int32_t p0, int n) {
  return n >= 0 && p0 >= 0 && (int64_t)p0 + n <= (int64_t)p.max_pages * p.page_size;
}

// One block per 128-key tile of a sequence (blockIdx.y = sequence), one warp per 16
// rows of it; a block whose tile no query of the chunk reads returns at once.
__global__ void __launch_bounds__(256) dequant_kernel(const PrefillParams p) {
  const int b = blockIdx.y;
  const int tile = blockIdx.x;
  const int lane = threadIdx.x & 31;
  const int32_t p0 = p.prefix_len[b];
  const SeqRows sr = seq_rows(p, b);
  const bool ok = seq_ok(p, p0, sr.n);
  if (!ok) {
    if (tile == 0 && threadIdx.x == 0 && p.err) atomicOr(p.err, CAI_DEVERR_LENGTH);
    return;
  }
  if (sr.n == 0) return;  // no new tokens (or a one-token row decoded elsewhere): nothing attends
  const int len = p0 + sr.n;
  if (tile * kKeys >= len) return;  // never read
  // Keys before every window of the chunk are never attended: rows of their tile get
  // zeros (masked later) and their pages are not read, so a local buffer may have
  // recycled them.
  const int lo_min = p.window > 0 ? max(0, p0 + 1 - p.window) : 0;
  if (tile < lo_min / kKeys) return;  // before every window, whole tile
  for (int rr = threadIdx.x >> 5; rr < kKeys; rr += blockDim.x >> 5) {
    const int t = tile * kKeys + rr;
    const int64_t row = (int64_t)b * p.kt_rows + t;
    uint32_t kw = 0, vw = 0;
    float ksc = 0.0f, vsc = 0.0f;
    if (t < len && t >= lo_min) {
      const int P = p.page_size;
      const int32_t page = p.table[(int64_t)b * p.max_pages + t / P];
      if (page >= 0 && page < p.num_pages) {
        const int slot = t % P;
        const uint8_t* pg = p.pages + (int64_t)page * page_bytes(P);
        kw = reinterpret_cast<const uint32_t*>(pg + slot * kHeadDim)[lane];
        const uint8_t* vcol = pg + P * kHeadDim + slot;  // channel-major V block: channel c at c * P
#pragma unroll
        for (int e = 0; e < 4; ++e) vw |= (uint32_t)vcol[(lane * 4 + e) * P] << (8 * e);
        const float* sc = reinterpret_cast<const float*>(pg + 2 * P * kHeadDim);
        ksc = sc[slot] * p.scale_log2;
        vsc = sc[P + slot];
      } else if (lane == 0 && p.err) {
        atomicOr(p.err, CAI_DEVERR_PAGE);
      }
    }
    // int8 -> bf16 (K) and int8 -> fp16 (V): exact for |code| <= 127.
    uint16_t kb[4], vh[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float kf = (float)(int8_t)(kw >> (8 * e));
      const float vf = (float)(int8_t)(vw >> (8 * e));
      kb[e] = (uint16_t)(__float_as_uint(kf) >> 16);  // small integers: the top half is exact
      const __half hv = __float2half_rn(vf * vsc);  // V scale applied here: P needs no per-key factor
      vh[e] = *reinterpret_cast<const uint16_t*>(&hv);
    }
    const int64_t off = row * kHeadDim + lane * 4;
    *reinterpret_cast<uint2*>(p.kb + off) = make_uint2(kb[0] | ((uint32_t)kb[1] << 16), kb[2] | ((uint32_t)kb[3] << 16));
    *reinterpret_cast<uint2*>(p.vh + off) = make_uint2(vh[0] | ((uint32_t)vh[1] << 16), vh[2] | ((uint32_t)vh[3] << 16));
    if (lane == 0) p.ks[row] = ksc;
  }
}

__device__ __forceinline__ void tma_load_rows128(void* dst, const CUtensorMap* map, int row, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], "
      "[%5];" ::"r"(smem_addr(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(0), "r"(row), "r"(0), "r"(smem_addr(bar))
      : "memory");
}

// One work item: a pair of q-tiles (256 consecutive (token, head) rows) of one
// sequence.  ok = false: no MMA work; the softmax groups then write zeros to the
// item's rows below `rows` (an invalid sequence) or nothing (rows beyond the chunk).
struct PItem {
  int b, row0, kt0, nkt;
  int64_t qrow0;  // first packed new-token row of the sequence
  int rows;       // (token, head) rows of the sequence, 0 if its offsets are invalid
  bool ok;
  int piece;      // -1: the whole key range; otherwise the piece's slot in piece_o / piece_lse
};

__device__ __forceinline__ PItem prefill_item(const PrefillParams& p, int idx) {
  PItem it;
  int pair = idx, piece = -1;
  if (idx >= p.full_items) {
    const int t = idx - p.full_items;
    pair = p.full_items + t / p.pieces;
    piece = t % p.pieces;
    it.piece = t;
  } else {
    it.piece = -1;
  }
  it.b = pair / p.pairs;
  it.row0 = (pair - it.b * p.pairs) * (kQT * kRows);
  const int32_t p0 = p.prefix_len[it.b];
  const SeqRows sr = seq_rows(p, it.b);
  it.qrow0 = sr.r0;
  it.rows = sr.n > 0 ? sr.n * p.num_heads : 0;
  it.ok = seq_ok(p, p0, sr.n) && it.row0 < it.rows;
  if (!it.ok) {
    it.kt0 = it.nkt = 0;
    return it;
  }
  const int i0 = it.row0 >> p.log2_heads;
  const int i_last = min((it.row0 + kQT * kRows - 1) >> p.log2_heads, sr.n - 1);
  const int kv_hi = p0 + i_last + 1;
  const int kv_lo = p.window > 0 ? max(0, p0 + i0 + 1 - p.window) : 0;
  it.kt0 = kv_lo / kKeys;
  it.nkt = (kv_hi - 1) / kKeys - it.kt0 + 1;
  if (piece >= 0) {  // key tiles [per * piece, per * (piece + 1)) of the pair's range
    const int per = (it.nkt + p.pieces - 1) / p.pieces;
    const int a = min(it.nkt, per * piece), e = min(it.nkt, per * (piece + 1));
    it.kt0 += a;
    it.nkt = e - a;
  }
  return it;
}

// Operand tiles in shared memory: element (r, k) of a 128x128 16-bit tile at
// (k/8)*2048 + r*16 + (k%8)*2 -- the order a [16 chunks][128 rows][8] TMA box
// writes.  As a K-major operand: LBO = 2048 (next 8 k), SBO = 128 (next 8 rows).
// As an MN-major operand (rows = K, k = N): LBO = 128, SBO = 2048.
//
// Persistent CTAs, one per SM, each taking pairs of q-tiles in turn.  Roles:
// warp 0 loads K/V tiles (TMA tensor copies) into a 2-stage ring; warp 1
// issues the MMAs in the order S0(j) S1(j) | PV0(j) S0(j+1) PV1(j) S1(j+1) ...
// so that each softmax group works on one tile while the tensor core runs the
// other group's MMAs; warps 2-5 and 6-9 run the softmax of q-tile 0 and 1 (one
// thread per row) and write the outputs.
__global__ void __launch_bounds__(kThreads, 1) prefill_kernel(const PrefillParams p,
                                                              const __grid_constant__ CUtensorMap kmap,
                                                              const __grid_constant__ CUtensorMap vmap) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kOffBars);
  uint64_t* k_full = bars;                     // [kStages] producer -> MMA (tx bytes)
  uint64_t* k_empty = bars + kStages;          // [kStages] MMA commit after both S of the tile
  uint64_t* v_full = bars + 2 * kStages;       // [kStages] producer -> MMA, softmax (V and K scales)
  uint64_t* v_empty = bars + 3 * kStages;      // [kStages] MMA commit after both PVs of the tile
  uint64_t* q_full = bars + 4 * kStages;       // [kQT] softmax group -> MMA (4 warps)
  uint64_t* s_full = q_full + kQT;             // [kQT] MMA commit after S
  uint64_t* p_full = s_full + kQT;             // [kQT] softmax -> MMA (4 warps)
  uint64_t* pv_done = p_full + kQT;            // [kQT] MMA commit after PV
  uint64_t* o_full = pv_done + kQT;            // [kQT] MMA commit after an item's last PV
  uint64_t* o_empty = o_full + kQT;            // [kQT] softmax -> MMA after reading O (4 warps)
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kOffMisc);
  volatile WaitState* const wctl = reinterpret_cast<volatile WaitState*>(smem + kOffMisc + 8);
  volatile int32_t* abort_flag = &wctl->abort;
  uint64_t* mma_drain = o_empty + kQT;         // the MMA issuer's last commit, at exit

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int Hq = p.num_heads;
  const int num_items = p.num_items;

  if (warp == 0) tmem_alloc(tmem_slot, kTmemCols);
  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&k_full[s], 1);
      mbar_init(&k_empty[s], 1);
      mbar_init(&v_full[s], 1);
      mbar_init(&v_empty[s], 1);
    }
    for (int q = 0; q < kQT; ++q) {
      mbar_init(&q_full[q], 4);
      mbar_init(&s_full[q], 1);
      mbar_init(&p_full[q], 4);
      mbar_init(&pv_done[q], 1);
      mbar_init(&o_full[q], 1);
      mbar_init(&o_empty[q], 4);
    }
    mbar_init(mma_drain, 1);
    *abort_flag = 0;
    wctl->limit_ns = p.wait_ns;
    fence_barrier_init();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp < 4) {
   setmaxnreg_dec<kRegsCtl>();
   if (warp == 0) {
    // ------------------------------------------------------------ K/V producer
    if (lane == 0) {
      int g = 0, gk = 0, gv = 0;  // tiles; tiles whose K and V loads were issued (or dropped)
      for (int idx = blockIdx.x; idx < num_items && !*abort_flag; idx += gridDim.x) {
        const PItem it = prefill_item(p, idx);
        const int64_t seq_row0 = (int64_t)it.b * p.kt_rows;
        for (int j = 0; j < it.nkt; ++j, ++g) {
          const int s = g % kStages;
          const int64_t row = seq_row0 + (int64_t)(it.kt0 + j) * kKeys;
          if (g >= kStages && !mbar_wait_abortable(&k_empty[s], ((g / kStages) - 1) & 1, wctl)) break;
          if (g != p.drop_stage) {  // (fault injection: that K tile is never loaded)
            mbar_arrive_expect_tx(&k_full[s], kTileBytes);
            tma_load_rows128(smem + kOffK + s * kTileBytes, &kmap, (int)row, &k_full[s]);
          }
          gk = g + 1;
          if (g >= kStages && !mbar_wait_abortable(&v_empty[s], ((g / kStages) - 1) & 1, wctl)) break;
          uint8_t* vs = smem + kOffV + s * kVSlotBytes;
          mbar_arrive_expect_tx(&v_full[s], kVSlotBytes);
          tma_load_rows128(vs, &vmap, (int)row, &v_full[s]);
          bulk_g2s(vs + kTileBytes, p.ks + row, kKeys * 4, &v_full[s]);
          gv = g + 1;
        }
      }
      // Every slot this producer armed has landed before the CTA goes away, whatever
      // happened to the other roles (copies into a CTA's shared memory must not outlive it).
      for (int i = gk > kStages ? gk - kStages : 0; i < gk; ++i)
        if (i != p.drop_stage) mbar_wait_drain(&k_full[i % kStages], (i / kStages) & 1);
      for (int i = gv > kStages ? gv - kStages : 0; i < gv; ++i) mbar_wait_drain(&v_full[i % kStages], (i / kStages) & 1);
    }
   } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc_s = idesc_bf16_f32(kRows, kKeys, 0, 0);
      constexpr uint32_t idesc_o = idesc_f16_f32(kRows, kHeadDim, 0, 1);
      const uint32_t qa0 = smem_addr(smem + kOffQ);
      int g = 0, n = 0;
      auto issue_s = [&](int q, int gg) {
        const uint32_t ka = smem_addr(smem + kOffK + (gg % kStages) * kTileBytes);
        const uint32_t qa = qa0 + q * kRows * kHeadDim * 2;
#pragma unroll
        for (int ks = 0; ks < kHeadDim / 16; ++ks)
          mma_f16_ss(tmem + q * 256, smem_desc(qa + ks * 4096, 2048, 128), smem_desc(ka + ks * 4096, 2048, 128),
                     idesc_s, ks > 0);
        mma_commit(&s_full[q]);
      };
      auto issue_pv = [&](int q, int gg, bool first) {
        const uint32_t va = smem_addr(smem + kOffV + (gg % kStages) * kVSlotBytes);
#pragma unroll
        for (int ks = 0; ks < kKeys / 16; ++ks)
          mma_f16_ts(tmem + q * 256 + 128, tmem + q * 256 + ks * 8, smem_desc(va + ks * 256, 128, 2048), idesc_o,
                     (!first || ks > 0) ? 1u : 0u);
        mma_commit(&pv_done[q]);
      };
      for (int idx = blockIdx.x; idx < num_items && !*abort_flag; idx += gridDim.x) {
        const PItem it = prefill_item(p, idx);
        if (!it.ok || it.nkt == 0) continue;  // no MMA work; the softmax groups write its zeros
        bool ok = mbar_wait_abortable(&q_full[0], n & 1, wctl) && mbar_wait_abortable(&q_full[1], n & 1, wctl);
        for (int j = 0; j < it.nkt && ok; ++j, ++g) {
          const int s = g % kStages;
          if (j == 0) {
            if (!mbar_wait_abortable(&k_full[s], (g / kStages) & 1, wctl)) break;
            tc_fence_after();
            issue_s(0, g);
            issue_s(1, g);
            mma_commit(&k_empty[s]);
          }
          const bool more = j + 1 < it.nkt;
          for (int q = 0; q < kQT; ++q) {
            if (!mbar_wait_abortable(&p_full[q], g & 1, wctl)) {
              ok = false;
              break;
            }
            if (j == 0 && n > 0 && !mbar_wait_abortable(&o_empty[q], (n - 1) & 1, wctl)) {
              ok = false;
              break;
            }
            if (q == 0 && !mbar_wait_abortable(&v_full[s], (g / kStages) & 1, wctl)) {
              ok = false;
              break;
            }
            tc_fence_after();
            issue_pv(q, g, j == 0);
            if (q == kQT - 1) mma_commit(&v_empty[s]);
            if (!more) mma_commit(&o_full[q]);
            if (more) {
              if (q == 0 && !mbar_wait_abortable(&k_full[(g + 1) % kStages], ((g + 1) / kStages) & 1, wctl)) {
                ok = false;
                break;
              }
              tc_fence_after();
              issue_s(q, g + 1);
              if (q == kQT - 1) mma_commit(&k_empty[(g + 1) % kStages]);
            }
          }
        }
        if (!ok) break;
        ++n;
      }
      // The issued MMAs have completed before tensor memory is freed.
      mma_commit(mma_drain);
      mbar_wait_drain(mma_drain, 0);
    }
   }
  } else {
    setmaxnreg_inc<kRegsSoft>();
    // ------------------------------------------------------------ softmax groups
    const int q = (warp - 4) >> 2;          // q-tile of this group
    const int quarter = warp & 3;           // TMEM lane quarter
    const int r = quarter * 32 + lane;      // row within the q-tile
    const uint32_t t_lane = (uint32_t)(quarter * 32) << 16;
    const uint32_t scol = (uint32_t)q * 256, ocol = scol + 128;
    uint8_t* qs = smem + kOffQ + q * kRows * kHeadDim * 2;
    // Each warp decides alone (its waits and its abort reads agree in all lanes); the
    // warps of a group meet only at mbarriers, so one that stops early strands nobody.
    int g = 0, n = 0;
    for (int idx = blockIdx.x; idx < num_items && !abort_seen_warp(wctl); idx += gridDim.x) {
      const PItem it = prefill_item(p, idx);
      const int64_t row = it.row0 + q * kRows + r;  // (token, head) row within the sequence
      const bool my_row = row < it.rows;
      const int my_i = (int)(row >> p.log2_heads), my_h = (int)(row & (Hq - 1));
      float* out_row = p.out + ((it.qrow0 + my_i) * Hq + my_h) * kHeadDim;
      if (!it.ok) {  // invalid sequence (flagged by the dequant pass): 0 / -inf; beyond the chunk: nothing
        if (my_row) {
          for (int d = 0; d < kHeadDim; d += 4)
            *reinterpret_cast<float4*>(out_row + d) = make_float4(0.f, 0.f, 0.f, 0.f);
          if (p.lse_out) p.lse_out[(it.qrow0 + my_i) * Hq + my_h] = -INFINITY;
        }
        continue;  // no MMA work for this item
      }
      // A piece's partial output row (normalised) and log2-sum-exp, for the merge.
      float* part_row = it.piece >= 0 ? p.piece_o + ((int64_t)it.piece * (kQT * kRows) + q * kRows + r) * kHeadDim
                                       : nullptr;
      if (it.nkt == 0) {  // a piece with no key tiles (no MMA work): weight zero in the merge
        for (int d = 0; d < kHeadDim; d += 4)
          *reinterpret_cast<float4*>(part_row + d) = make_float4(0.f, 0.f, 0.f, 0.f);
        p.piece_lse[(int64_t)it.piece * (kQT * kRows) + q * kRows + r] = -INFINITY;
        continue;
      }
      // This row's query (bf16), zero beyond the chunk.
      {
        const uint4* src = reinterpret_cast<const uint4*>(p.q + (it.qrow0 * Hq + row) * kHeadDim);
#pragma unroll
        for (int c = 0; c < 16; ++c)
          *reinterpret_cast<uint4*>(qs + c * 2048 + r * 16) = my_row ? src[c] : make_uint4(0, 0, 0, 0);
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(&q_full[q]);
      const int32_t p0 = p.prefix_len[it.b];
      const int q_pos = p0 + my_i;
      const int k_lo = p.window > 0 ? max(0, q_pos + 1 - p.window) : 0;
      float m_ref = -INFINITY, l_sum = 0.0f;
      bool ok = true;
      for (int j = 0; j < it.nkt; ++j, ++g) {
        const int s = g % kStages;
        ok = mbar_wait_warp(&s_full[q], g & 1, wctl) &&
             mbar_wait_warp(&v_full[s], (g / kStages) & 1, wctl);
        if (!ok) break;
        tc_fence_after();
        const float* kscale = reinterpret_cast<const float*>(smem + kOffV + s * kVSlotBytes + kTileBytes);
        const int key0 = (it.kt0 + j) * kKeys;
        // z = logit (log2 units) minus the row's reference maximum, one FFMA per key.
        const float m_use = m_ref == -INFINITY ? 0.0f : m_ref;
        float z[kKeys];
#pragma unroll
        for (int c = 0; c < kKeys; c += 32) {
          uint32_t rr[32];
          tmem_ld_32x32b_x32(tmem + t_lane + scol + c, rr);
          tmem_wait_ld();
#pragma unroll
          for (int e = 0; e < 32; e += 4) {
            const float4 a = *reinterpret_cast<const float4*>(kscale + c + e);
            z[c + e] = fmaf(__uint_as_float(rr[e]), a.x, -m_use);
            z[c + e + 1] = fmaf(__uint_as_float(rr[e + 1]), a.y, -m_use);
            z[c + e + 2] = fmaf(__uint_as_float(rr[e + 2]), a.z, -m_use);
            z[c + e + 3] = fmaf(__uint_as_float(rr[e + 3]), a.w, -m_use);
          }
        }
        if (!(key0 >= k_lo && key0 + kKeys - 1 <= q_pos)) {
#pragma unroll
          for (int c = 0; c < kKeys; ++c) {
            const int key = key0 + c;
            if (key < k_lo || key > q_pos) z[c] = -INFINITY;
          }
        }
        float mx4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
        for (int c = 0; c < kKeys; c += 8) {
          mx4[0] = fmax3(mx4[0], z[c], z[c + 1]);
          mx4[1] = fmax3(mx4[1], z[c + 2], z[c + 3]);
          mx4[2] = fmax3(mx4[2], z[c + 4], z[c + 5]);
          mx4[3] = fmax3(mx4[3], z[c + 6], z[c + 7]);
        }
        const float mx = fmaxf(fmaxf(mx4[0], mx4[1]), fmaxf(mx4[2], mx4[3]));
        // Raise the reference when the row has none yet, or a logit exceeds it by 2^8.
        const bool raise = m_ref == -INFINITY ? mx > -INFINITY : mx > kRescaleThreshold;
        const float alpha = raise ? ex2_approx(m_ref - (m_use + mx)) : 1.0f;  // 0 when there was no reference
        if (j > 0 && __any_sync(0xffffffffu, raise)) {
          ok = mbar_wait_warp(&pv_done[q], (g - 1) & 1, wctl);
          if (ok) {
            tc_fence_after();
#pragma unroll
            for (int c = 0; c < kHeadDim; c += 32) {
              uint32_t o[32];
              tmem_ld_32x32b_x32(tmem + t_lane + ocol + c, o);
              tmem_wait_ld();
#pragma unroll
              for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
              tmem_st_32x32b_x32(tmem + t_lane + ocol + c, o);
            }
            tmem_wait_st();
          }
        }
        if (raise) {
          l_sum *= alpha;
          m_ref = m_use + mx;
#pragma unroll
          for (int c = 0; c < kKeys; ++c) z[c] -= mx;
        }
        float l4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int c = 0; c < kKeys; c += 64) {
          uint32_t pw[32];
#pragma unroll
          for (int e = 0; e < 64; e += 4) {
            const float e0 = ex2_approx(z[c + e]), e1 = ex2_approx(z[c + e + 1]);
            const float e2 = ex2_approx(z[c + e + 2]), e3 = ex2_approx(z[c + e + 3]);
            l4[0] += e0;
            l4[1] += e1;
            l4[2] += e2;
            l4[3] += e3;
            pw[e / 2] = pack_f16x2(e0, e1);
            pw[e / 2 + 1] = pack_f16x2(e2, e3);
          }
          tmem_st_32x32b_x32(tmem + t_lane + scol + c / 2, pw);
        }
        l_sum += (l4[0] + l4[1]) + (l4[2] + l4[3]);
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&p_full[q]);
        if (!ok) break;
      }
      if (!ok) break;
      if (!mbar_wait_warp(&o_full[q], n & 1, wctl)) break;
      tc_fence_after();
      const float inv = l_sum > 0.0f ? 1.0f / l_sum : 0.0f;
      float* dst = part_row ? part_row : out_row;
#pragma unroll
      for (int c = 0; c < kHeadDim; c += 32) {
        uint32_t o[32];
        tmem_ld_32x32b_x32(tmem + t_lane + ocol + c, o);
        tmem_wait_ld();
        if (my_row) {
#pragma unroll
          for (int e = 0; e < 32; e += 4)
            *reinterpret_cast<float4*>(dst + c + e) =
                make_float4(__uint_as_float(o[e]) * inv, __uint_as_float(o[e + 1]) * inv,
                            __uint_as_float(o[e + 2]) * inv, __uint_as_float(o[e + 3]) * inv);
        }
      }
      const float lse2 = l_sum > 0.0f ? m_ref + __log2f(l_sum) : -INFINITY;
      if (part_row) {
        if (my_row) p.piece_lse[(int64_t)it.piece * (kQT * kRows) + q * kRows + r] = lse2;
      } else if (my_row && p.lse_out) {
        p.lse_out[(it.qrow0 + my_i) * Hq + my_h] = lse2 * kLn2;
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&o_empty[q]);
      ++n;
    }
  }
  tc_fence_before();
  __syncthreads();
  if (tid == 0 && *abort_flag && p.err) atomicOr(p.err, CAI_DEVERR_TIMEOUT);
  if (warp == 0) tmem_dealloc(tmem, kTmemCols);
}

// One warp per (split pair, row): merge the pair's pieces by their log-sum-exp,
// out = sum_j 2^(lse_j - M) o_j / sum_j 2^(lse_j - M), into the row's output.
__global__ void __launch_bounds__(256) combine_pieces_kernel(const PrefillParams p) {
  grid_dependency_wait();
  grid_launch_dependents();
  const int64_t w = (blockIdx.x * (int64_t)blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  const int split_pairs = (p.num_items - p.full_items) / p.pieces;
  if (w >= (int64_t)split_pairs * (kQT * kRows)) return;
  const int sp = (int)(w / (kQT * kRows)), r = (int)(w % (kQT * kRows));
  const PItem it = prefill_item(p, p.full_items + sp * p.pieces);
  const int64_t row = it.row0 + r;
  if (!it.ok || row >= it.rows) return;  // invalid sequence (its rows hold zeros) or past the chunk
  const int Hq = p.num_heads;
  const int my_i = (int)(row >> p.log2_heads), my_h = (int)(row & (Hq - 1));
  const int64_t t0 = (int64_t)sp * p.pieces;
  const float lj = lane < p.pieces ? p.piece_lse[(t0 + lane) * (kQT * kRows) + r] : -INFINITY;
  float M = lj;
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
  const float wj = (M == -INFINITY || lane >= p.pieces) ? 0.0f : ex2_approx(lj - M);
  float wsum = wj;
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) wsum += __shfl_xor_sync(0xffffffffu, wsum, o);
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int j = 0; j < p.pieces; ++j) {
    const float wt = __shfl_sync(0xffffffffu, wj, j);
    const float4 o = reinterpret_cast<const float4*>(p.piece_o + ((t0 + j) * (kQT * kRows) + r) * kHeadDim)[lane];
    acc.x = fmaf(wt, o.x, acc.x);
    acc.y = fmaf(wt, o.y, acc.y);
    acc.z = fmaf(wt, o.z, acc.z);
    acc.w = fmaf(wt, o.w, acc.w);
  }
  const float inv = wsum > 0.0f ? 1.0f / wsum : 0.0f;
  reinterpret_cast<float4*>(p.out + ((it.qrow0 + my_i) * Hq + my_h) * kHeadDim)[lane] =
      make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv);
  if (p.lse_out && lane == 0)
    p.lse_out[(it.qrow0 + my_i) * Hq + my_h] = wsum > 0.0f ? (M + __log2f(wsum)) * kLn2 : -INFINITY;
}

// A [rows][128] 16-bit row-major matrix seen as (8 elements, rows, 16 chunks)
// so that a (8, 128, 16) box lands in shared memory as [chunk][row][8].
bool encode_rows128(CUtensorMap* map, const void* base, uint64_t rows) {
  auto fn = tensor_map_encoder();
  if (!fn) return false;
  cuuint64_t dims[3] = {8, rows, 16};
  cuuint64_t strides[2] = {kHeadDim * 2, 16};
  cuuint32_t box[3] = {8, (cuuint32_t)kRows, 16};
  cuuint32_t estr[3] = {1, 1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT16, 3, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

// Partial outputs of the split last wave: at most one piece per CTA of the grid.
static int64_t piece_bytes() { return (int64_t)num_sms() * (kQT * kRows) * (kHeadDim + 1) * 4; }

size_t prefill_workspace_bytes(int32_t batch, int32_t max_pages_per_seq, int32_t page_size) {
  const int64_t kt = ((int64_t)max_pages_per_seq * page_size + kKeys - 1) / kKeys * kKeys;
  const int64_t rows = (int64_t)batch * kt;
  const int64_t a = ((rows * kHeadDim * 2 + 255) / 256) * 256;
  const int64_t s = ((rows * 4 + 255) / 256) * 256;
  // ... and, last, the work-queue counters of the decode launch that takes a varlen batch's
  // one-token rows (see cai_mqa_prefill_varlen).
  return (size_t)(2 * a + 2 * s + ((piece_bytes() + 255) / 256) * 256 + kWorkspaceHeader);
}

// The piece region of a prefill workspace: the prefill kernel writes the last wave's
// partial outputs there, and a varlen call's decode launch, which runs before it on the
// same stream, may keep its split partials there.
void prefill_piece_region(void* workspace, int32_t batch, int32_t max_pages_per_seq, int32_t page_size,
                          void** region, size_t* bytes) {
  const int64_t kt = ((int64_t)max_pages_per_seq * page_size + kKeys - 1) / kKeys * kKeys;
  const int64_t rows = (int64_t)batch * kt;
  const int64_t a = ((rows * kHeadDim * 2 + 255) / 256) * 256;
  const int64_t s = ((rows * 4 + 255) / 256) * 256;
  *region = static_cast<uint8_t*>(workspace) + 2 * a + 2 * s;
  *bytes = (size_t)(((piece_bytes() + 255) / 256) * 256);
}

cudaError_t launch_prefill(const PrefillLaunch& L, cudaStream_t stream) {
  PrefillParams p;
  p.pages = L.pages;
  p.num_pages = L.num_pages;
  p.page_size = L.page_size;
  p.max_pages = L.max_pages;
  p.table = L.table;
  p.prefix_len = L.prefix_len;
  p.q = L.q;
  p.q_off = L.q_off;
  p.skip_single = L.q_off && L.skip_single ? 1 : 0;
  p.batch = L.batch;
  p.n_new = L.n_new;
  p.total_new = L.total_new;
  p.num_heads = L.num_heads;
  p.log2_heads = 31 - __builtin_clz((unsigned)L.num_heads);
  p.window = L.window;
  p.kt_rows = (int32_t)(((int64_t)L.max_pages * L.page_size + kKeys - 1) / kKeys * kKeys);
  p.pairs = (int32_t)(((int64_t)L.n_new * L.num_heads + kQT * kRows - 1) / (kQT * kRows));
  p.scale_log2 = L.scale_log2;
  p.wait_ns = wait_limit_ns();
  p.drop_stage = fault_drop_stage();
  const int64_t rows = (int64_t)L.batch * p.kt_rows;
  const int64_t a = ((rows * kHeadDim * 2 + 255) / 256) * 256;
  uint8_t* ws = static_cast<uint8_t*>(L.workspace);
  p.kb = reinterpret_cast<uint16_t*>(ws);
  p.vh = reinterpret_cast<uint16_t*>(ws + a);
  p.ks = reinterpret_cast<float*>(ws + 2 * a);
  const int64_t sbytes = ((rows * 4 + 255) / 256) * 256;
  p.piece_o = reinterpret_cast<float*>(ws + 2 * a + 2 * sbytes);
  p.piece_lse = p.piece_o + (int64_t)num_sms() * (kQT * kRows) * kHeadDim;
  p.out = L.out;
  p.lse_out = L.lse_out;
  p.err = L.err;

  CUtensorMap kmap, vmap;
  if (!encode_rows128(&kmap, p.kb, (uint64_t)rows) || !encode_rows128(&vmap, p.vh, (uint64_t)rows))
    return cudaErrorInvalidValue;

  dequant_kernel<<<dim3((unsigned)(p.kt_rows / kKeys), (unsigned)L.batch), 256, 0, stream>>>(p);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;

  static bool attr_set[64] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 64 && !attr_set[dev]) {
    // The register split inside the kernel assumes the launch register count.
    cudaFuncAttributes fa;
    e = cudaFuncGetAttributes(&fa, prefill_kernel);
    if (e != cudaSuccess) return e;
    if (fa.numRegs != kRegsLaunch) return cudaErrorInvalidDeviceFunction;
    e = cudaFuncSetAttribute(prefill_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    if (e != cudaSuccess) return e;
    attr_set[dev] = true;
  }
  // Work split: whole pairs in full waves of the persistent grid; the pairs of a partial
  // last wave are cut into `pieces` key ranges so that wave ends sooner (with r pairs
  // left over, pieces = grid / r, at most 4; the pieces of a pair are merged after).
  const int64_t pairs_total = (int64_t)L.batch * p.pairs;
  const int sms = num_sms();
  const int grid = (int)(pairs_total < sms ? pairs_total : sms);
  const int64_t rem = pairs_total % grid;
  int pieces = rem > 0 ? (int)(grid / rem) : 1;
  if (pieces > 4) pieces = 4;
  if (pieces < 2) pieces = 1;
  p.pieces = pieces;
  p.full_items = (int32_t)(pieces > 1 ? pairs_total - rem : pairs_total);
  p.num_items = (int32_t)(p.full_items + (pieces > 1 ? rem * pieces : 0));
  prefill_kernel<<<grid, kThreads, kSmemBytes, stream>>>(p, kmap, vmap);
  e = cudaGetLastError();
  if (e != cudaSuccess || pieces == 1) return e;
  const int64_t warps_c = rem * (kQT * kRows);
  return launch_pdl(combine_pieces_kernel, dim3((unsigned)((warps_c + 7) / 8)), dim3(256), 0, stream, p);
}

}  // namespace cai
