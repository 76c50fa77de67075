// Split-KV MQA decode over the int8 paged KV cache, and the log-sum-exp
// combine of the splits.
//
// What it computes (definition): for one query token per sequence and each
// query head h, softmax over the attended positions t of
//   z_t = softmax_scale * <q_h, s_k[t] * k_code[t]>
// and out_h = sum_t p_t * s_v[t] * v_code[t]  (Red Hat page, "Por que o cache
// KV existe"), where every head reads the same single K/V head (Multi-Query
// Attention) and a local layer attends only the last `window` positions
// (hybrid attention, technique table of "Character.AI: inference
// optimization", section 03).
//
// How.  A persistent kernel, one CTA per SM, walks a static list of work
// items (sequence, split) in 128-token tiles with five warp roles connected by
// mbarriers:
//  * producer (warp 0): one 1-D bulk copy (TMA engine) per page into a
//    3-stage ring; a page carries K codes, V codes and both scale rows and is
//    read once for all query heads.  Pages wholly outside the split (the part
//    of a local layer before its window) are never read;
//  * converters (warps 2-5): int8 codes -> fp16 (exact) into the canonical
//    no-swizzle tcgen05 operand layouts in shared memory (K K-major, V
//    MN-major), the per-token scales and mask into a small ring, and the
//    item's query (bf16 -> fp16) into tensor memory;
//  * MMA issuer (warp 1): S = Q K^T (tcgen05.mma kind::f16, M = 64 padded
//    heads, N = 128 tokens, K = 128, A from tensor memory) into a double-
//    buffered S, then O += P V (P from tensor memory, V from shared memory);
//  * softmax (warps 6-9, two threads per head): applies the per-token K scale
//    and softmax scale in fp32, keeps a reference maximum that is raised only
//    when a logit exceeds it by 2^8 (so O is rarely rescaled), scales P by the
//    per-token V scale, rounds it to fp16 into the S buffer it came from, and
//    at the end of an item writes the normalised partial output and its
//    log-sum-exp (or the final output when the sequence has one split).
#include "common.cuh"
#include "ptx.cuh"

namespace cai {
namespace {

constexpr int T = kDecodeTile;                 // 128 tokens per MMA tile
constexpr int RT = kRawTokens;                 // 64 tokens per raw stage
constexpr int NST = kDecodeStages;             // raw page stages
constexpr int kRawStageBytes = RT * 264;       // K, V and scales of 64 tokens
constexpr int kOp16Bytes = T * kHeadDim * 2;   // one fp16 operand tile (32 KB)
constexpr int kRing = 8;                       // work items published ahead by the producer
constexpr int kOffRaw = 0;
constexpr int kOffK16 = kOffRaw + NST * kRawStageBytes;  // K16[2]
constexpr int kOffV16 = kOffK16 + 2 * kOp16Bytes;        // V16[2]
constexpr int kOffScale = kOffV16 + 2 * kOp16Bytes;      // [2][3][T] floats: k scale, bias, v scale
constexpr int kOffBars = kOffScale + 2 * 3 * T * 4;
constexpr int kNumBars = 2 * NST + 2 * 2 /*k_full,v_full*/ + 2 * 2 /*s_full,p_full*/ + 2 /*v_free*/ + 2 /*o*/ +
                         2 * kRing;
constexpr int kOffMisc = kOffBars + 8 * kNumBars;        // tmem slot, abort flag, tile_full[2], page_ok[NST]
constexpr int kOffRing = kOffMisc + 64;                  // [kRing] published work items
constexpr int kRingInts = 16;                            // one ring entry: fields + first tile's page ids
constexpr int kOffXch = kOffRing + kRing * kRingInts * 4;    // [2 tiles][2 halves][64 rows] floats
constexpr int kSmemBytes = kOffXch + 3 * 2 * 64 * 4 + 1024;  // maxima [2][2][64] + sums [2][64]
// Warp roles, aligned to warpgroups so each group can resize its register file:
//   warpgroup 0: producer (warp 0), MMA issuer (warp 1), scheduler (warp 2), spare (warp 3)
//   warpgroups 1-2: converters (warps 4..11)
//   warpgroups 3-4: softmax (warps 12..19: two per TMEM lane quarter, each taking
//   half of a tile's tokens)
constexpr int kThreads = 640;
constexpr int kSchedWarp = 2;
constexpr int kConvWarp0 = 4;
constexpr int kConvWarps = 8;
constexpr int kSoftWarp0 = kConvWarp0 + kConvWarps;
constexpr int kSoftWarps = 8;
// Registers per thread: launched with 96 (20 warps: 5 per SM sub-partition,
// 5 * 32 * 96 = 15360 <= 16384), then 4 warps x 56 + 8 x 96 + 8 x 112:
// 128 * (56 + 2 * 96 + 2 * 112) = 60416 <= 640 * 96 = 61440.
constexpr int kRegsCtl = 56, kRegsConv = 96, kRegsSoft = 112;
constexpr int kRegsLaunch = 96;  // checked on the host before the first launch
constexpr int kNoPage = -2147483647 - 1;                 // a page the tile does not need
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColQ = 0;    // Q[2]: 64 columns each (128 fp16 channels as pairs)
constexpr uint32_t kColS = 128;  // S[2]: 128 columns each; P (fp16 pairs) overwrites the first 64
constexpr uint32_t kColO = 384;  // O: 128 columns
constexpr float kRescaleThreshold = 8.0f;  // log2 units: weights stay <= 2^8 between rescales
constexpr int kItemReaders = 2 + kConvWarps + kSoftWarps;  // producer, MMA, converters, softmax

// K-major no-swizzle operand with 128 channels: element (t, k) at
// (t/8)*2048 + (k/8)*128 + (t%8)*16 + (k%8)*2.
__device__ __forceinline__ uint32_t kmajor_off(int t, int k8) { return (t >> 3) * 2048 + k8 * 128 + (t & 7) * 16; }
// MN-major no-swizzle operand, T tokens along K and 128 channels along N:
// element (t, n) at (n/8)*(T*16) + (t/8)*128 + (t%8)*16 + (n%8)*2.
__device__ __forceinline__ uint32_t mnmajor_off(int t, int n8) { return n8 * (T * 16) + (t >> 3) * 128 + (t & 7) * 16; }

__device__ __forceinline__ void set_err(int32_t* err, int bits) {
  if (err) atomicOr(err, bits);
}

// A work item: one split of one sequence.  kind 0 = tiles to process,
// 1 = nothing to attend (split 0 writes out = 0, lse = -inf).
struct Item {
  int b, split, start, end, tile0, ntiles;
  bool direct;  // single split: write the final output
  int kind;
  bool invalid;
};

// Ring entry: [0] b, [1] split, [2] start, [3] end, [4] tile0, [5] ntiles,
// [6] flags (bit 0 direct, bit 1 invalid, bit 2 kind 1, bit 3 end of work),
// [8 .. 8 + T/P) page ids of the item's first tile (kNoPage where not needed).
__device__ __forceinline__ Item ring_item(const volatile int32_t* e, bool& done) {
  Item it;
  it.b = e[0];
  it.split = e[1];
  it.start = e[2];
  it.end = e[3];
  it.tile0 = e[4];
  it.ntiles = e[5];
  const int f = e[6];
  it.direct = f & 1;
  it.invalid = (f >> 1) & 1;
  it.kind = (f >> 2) & 1;
  done = (f >> 3) & 1;
  return it;
}

// Page id of page slot `ps` of tile `t` of an item, or kNoPage if the tile does not need it.
template <int P>
__device__ __forceinline__ int32_t tile_page(const DecodeParams& p, const Item& it, int t, int ps) {
  const int t0 = (it.tile0 + t) * T + ps * P;
  if (ps >= T / P || t0 + P <= it.start || t0 >= it.end) return (int32_t)kNoPage;
  return p.table[(int64_t)it.b * p.max_pages + t0 / P];
}

// kind 2 = an empty split, never published.
template <int P>
__device__ __forceinline__ Item make_item(const DecodeParams& p, int idx) {
  Item it;
  it.b = idx / p.plan.max_splits;
  it.split = idx - it.b * p.plan.max_splits;
  const SeqSplits sp = seq_splits(p.ctx_len[it.b], p.window, p.max_pages * P, p.plan.chunk);
  it.invalid = !sp.valid;
  it.direct = sp.nsplit == 1;
  it.ntiles = 0;
  it.start = it.end = it.tile0 = 0;
  if (sp.nsplit == 0) {
    it.kind = it.split == 0 ? 1 : 2;
    return it;
  }
  if (it.split >= sp.nsplit) {
    it.kind = 2;
    return it;
  }
  it.kind = 0;
  it.start = sp.lo + it.split * p.plan.chunk;
  it.end = min(sp.hi, it.start + p.plan.chunk);
  it.tile0 = it.start / T;
  it.ntiles = (it.end - 1) / T - it.tile0 + 1;
  return it;
}

template <int P>
__global__ void __launch_bounds__(kThreads, 1) decode_kernel(const DecodeParams p) {
  static_assert(kRegsCtl * 128 + kRegsConv * 256 + kRegsSoft * 256 <= kRegsLaunch * kThreads, "register split");
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* raw = smem + kOffRaw;
  uint8_t* k16 = smem + kOffK16;
  uint8_t* v16 = smem + kOffV16;
  float* scal = reinterpret_cast<float*>(smem + kOffScale);  // [2][3][T]
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kOffBars);
  uint64_t* raw_full = bars;              // [NST] producer -> converters (tx bytes)
  uint64_t* raw_empty = bars + NST;       // [NST] converters -> producer (4 warps)
  uint64_t* k_full = bars + 2 * NST;      // [2] converters -> MMA, softmax (4 warps)
  uint64_t* v_full = k_full + 2;          // [2] converters -> MMA (4 warps)
  uint64_t* s_full = v_full + 2;          // [2] MMA commit after S
  uint64_t* p_full = s_full + 2;          // [2] softmax -> MMA, converters (4 warps)
  uint64_t* v_free = p_full + 2;          // [2] MMA commit after PV
  uint64_t* o_full = v_free + 2;          // MMA commit after an item's last PV
  uint64_t* o_empty = o_full + 1;         // softmax -> MMA after reading O (4 warps)
  uint64_t* item_full = o_empty + 1;      // [kRing] producer -> readers
  uint64_t* item_empty = item_full + kRing;  // [kRing] readers -> producer
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kOffMisc);
  volatile int32_t* abort_flag = reinterpret_cast<volatile int32_t*>(smem + kOffMisc + 4);
  int32_t* tile_full = reinterpret_cast<int32_t*>(smem + kOffMisc + 8);               // [2]
  uint32_t* page_ok = reinterpret_cast<uint32_t*>(smem + kOffMisc + 16);             // [NST]
  volatile int32_t* ring = reinterpret_cast<volatile int32_t*>(smem + kOffRing);      // [kRing][kRingInts]

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int Hq = p.num_heads;
  const int num_items = p.batch * p.plan.max_splits;

  if (warp == 0) tmem_alloc(tmem_slot, kTmemCols);
  if (tid == 0) {
    for (int s = 0; s < NST; ++s) {
      mbar_init(&raw_full[s], 1);
      mbar_init(&raw_empty[s], kConvWarps);
    }
    for (int c = 0; c < 2; ++c) {
      mbar_init(&k_full[c], kConvWarps);
      mbar_init(&v_full[c], kConvWarps);
      mbar_init(&s_full[c], 1);
      mbar_init(&p_full[c], kSoftWarps);
      mbar_init(&v_free[c], 1);
    }
    mbar_init(o_full, 1);
    mbar_init(o_empty, kSoftWarps);
    for (int r = 0; r < kRing; ++r) {
      mbar_init(&item_full[r], 1);
      mbar_init(&item_empty[r], kItemReaders);
    }
    *abort_flag = 0;
    fence_barrier_init();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  // Item k of this CTA as published by the scheduler warp; every reader warp
  // waits for it, copies it and releases the slot.
  auto next_item = [&](int k, bool& done, int32_t* first_ids = nullptr) -> Item {
    const int slot = k % kRing;
    Item it = {};
    if (!mbar_wait_abortable(&item_full[slot], (k / kRing) & 1, abort_flag)) {
      done = true;
      return it;
    }
    it = ring_item(ring + slot * kRingInts, done);
    if (first_ids) *first_ids = lane < T / P ? (int32_t)ring[slot * kRingInts + 8 + lane] : (int32_t)kNoPage;
    __syncwarp();
    if (lane == 0) mbar_arrive(&item_empty[slot]);
    return it;
  };

  if (warp < kConvWarp0) {
   setmaxnreg_dec<kRegsCtl>();
   if (warp == kSchedWarp) {
    // ------------------------------------------------------------ scheduler
    // Takes work items from the global queue, decodes them and publishes them,
    // up to kRing ahead of the roles that consume them.
    int k = 0;
    while (true) {
      int idx = 0;
      if (lane == 0) idx = (int)atomicAdd(&p.queue[0], 1u);
      idx = __shfl_sync(0xffffffffu, idx, 0);
      const bool done = idx >= num_items;
      Item it = {};
      int32_t id = (int32_t)kNoPage;
      if (!done) {
        it = make_item<P>(p, idx);
        if (it.kind == 2) continue;  // an empty split: nobody needs to hear of it
        if (it.kind == 0) {
          id = tile_page<P>(p, it, 0, lane);
          // Warm L2 with the item's block-table entries (32 ids per 128-byte line, one line per lane).
          const int first = it.start / P, last = (it.end - 1) / P;
          const int32_t* row = p.table + (int64_t)it.b * p.max_pages;
          for (int pg = (first & ~31) + lane * 32; pg <= last; pg += 32 * 32) prefetch_l2(row + pg);
        }
      }
      const int slot = k % kRing;
      if (k >= kRing && !mbar_wait_abortable(&item_empty[slot], ((k / kRing) - 1) & 1, abort_flag)) break;
      volatile int32_t* e = ring + slot * kRingInts;
      if (lane < T / P) e[8 + lane] = id;
      if (lane == 0) {
        if (!done) {
          e[0] = it.b;
          e[1] = it.split;
          e[2] = it.start;
          e[3] = it.end;
          e[4] = it.tile0;
          e[5] = it.ntiles;
          e[6] = (it.direct ? 1 : 0) | (it.invalid ? 2 : 0) | (it.kind == 1 ? 4 : 0);
        } else {
          e[6] = 8;
        }
      }
      __syncwarp();
      if (lane == 0) {
        __threadfence_block();
        mbar_arrive(&item_full[slot]);
      }
      ++k;
      if (done) break;
    }
    // The last CTA to finish fetching leaves the queue counters at zero for the next call.
    if (lane == 0 && atomicAdd(&p.queue[1], 1u) == gridDim.x - 1) {
      atomicExch(&p.queue[0], 0u);
      atomicExch(&p.queue[1], 0u);
    }
  } else if (warp == 0) {
    // ------------------------------------------------------------ producer
    // Page ids are fetched one tile ahead by the warp's lanes (lane i: page slot i).
    const uint64_t policy = policy_evict_first();
    int r = 0, k = 0;
    while (true) {
      bool done = false;
      int32_t ids = kNoPage;
      const Item it = next_item(k++, done, &ids);
      if (done || *abort_flag) break;
      if (it.kind != 0) continue;
      bool ok = true;
      int32_t ids_n1 = (1 < it.ntiles) ? tile_page<P>(p, it, 1, lane) : (int32_t)kNoPage;
      for (int t = 0; t < it.ntiles && ok; ++t) {
        const int32_t ids_n2 = (t + 2 < it.ntiles) ? tile_page<P>(p, it, t + 2, lane) : (int32_t)kNoPage;
        for (int hf = 0; hf < 2; ++hf, ++r) {
          const int s = r % NST;
          if (r >= NST && !mbar_wait_abortable(&raw_empty[s], ((r / NST) - 1) & 1, abort_flag)) {
            ok = false;
            break;
          }
          int32_t pid[RT / P];
#pragma unroll
          for (int ps = 0; ps < RT / P; ++ps) pid[ps] = __shfl_sync(0xffffffffu, ids, hf * (RT / P) + ps);
          if (lane == 0) {
            uint32_t okm = 0, bytes = 0;
#pragma unroll
            for (int ps = 0; ps < RT / P; ++ps) {
              if (pid[ps] == kNoPage) continue;
              if (pid[ps] < 0 || pid[ps] >= p.num_pages) {
                set_err(p.err, CAI_DEVERR_PAGE);
                continue;
              }
              okm |= 1u << ps;
              bytes += page_bytes(P);
            }
            page_ok[s] = okm;
            mbar_arrive_expect_tx(&raw_full[s], bytes);
#pragma unroll
            for (int ps = 0; ps < RT / P; ++ps) {
              if (!(okm & (1u << ps))) continue;
              bulk_g2s_hint(raw + s * kRawStageBytes + ps * page_bytes(P),
                            p.pages + (int64_t)pid[ps] * page_bytes(P), page_bytes(P), &raw_full[s], policy);
            }
          }
          __syncwarp();
        }
        ids = ids_n1;
        ids_n1 = ids_n2;
      }
      if (!ok) break;
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    constexpr uint32_t idesc_s = idesc_f16_f32(kDecodeRows, T, 0, 0);
    constexpr uint32_t idesc_o = idesc_f16_f32(kDecodeRows, kHeadDim, 0, 1);
    const uint32_t k16a = smem_addr(k16), v16a = smem_addr(v16);
    int g = 0, item_n = 0, k = 0;
    bool have_prev = false, prev_first = false, prev_last = false;
    int prev_item_n = 0;
    auto issue_pv = [&](int gp) {
      const int c = gp & 1;
      if (!mbar_wait_abortable(&p_full[c], (gp >> 1) & 1, abort_flag)) return;
      if (!mbar_wait_abortable(&v_full[c], (gp >> 1) & 1, abort_flag)) return;
      if (prev_first && prev_item_n > 0 && !mbar_wait_abortable(o_empty, (prev_item_n - 1) & 1, abort_flag)) return;
      tc_fence_after();
      if (lane == 0) {
#pragma unroll
        for (int ks = 0; ks < T / 16; ++ks)
          mma_f16_ts(tmem + kColO, tmem + kColS + c * 128 + ks * 8,
                     smem_desc(v16a + c * kOp16Bytes + ks * 256, 128, T * 16), idesc_o,
                     (!prev_first || ks > 0) ? 1u : 0u);
        mma_commit(&v_free[c]);
        if (prev_last) mma_commit(o_full);
      }
      __syncwarp();
    };
    while (true) {
      bool done = false;
      const Item it = next_item(k++, done);
      if (done) break;
      if (it.kind != 0) continue;
      bool ok = true;
      for (int t = 0; t < it.ntiles; ++t, ++g) {
        const int c = g & 1;
        if (!mbar_wait_abortable(&k_full[c], (g >> 1) & 1, abort_flag)) {
          ok = false;
          break;
        }
        tc_fence_after();
        if (lane == 0) {
          const uint32_t qcol = kColQ + (item_n & 1) * 64;
#pragma unroll
          for (int ks = 0; ks < kHeadDim / 16; ++ks)
            mma_f16_ts(tmem + kColS + c * 128, tmem + qcol + ks * 8,
                       smem_desc(k16a + c * kOp16Bytes + ks * 256, 128, 2048), idesc_s, ks > 0 ? 1u : 0u);
          mma_commit(&s_full[c]);
        }
        __syncwarp();
        if (have_prev) issue_pv(g - 1);
        have_prev = true;
        prev_first = t == 0;
        prev_last = t == it.ntiles - 1;
        prev_item_n = item_n;
      }
      if (!ok) break;
      ++item_n;
    }
    if (have_prev && !*abort_flag) issue_pv(g - 1);
   }
  } else if (warp < kSoftWarp0) {
    setmaxnreg_dec<kRegsConv>();
    // ------------------------------------------------------------ converters
    const int ctid = tid - kConvWarp0 * 32;  // 0 .. 32*kConvWarps-1
    const int quarter = warp & 3;            // TMEM lanes this warp may touch
    const bool q_warp = warp < kConvWarp0 + 4;  // one warp per lane quarter stores the query
    constexpr int kUnits = (T * 8) / (32 * kConvWarps);  // 16-byte units per thread per operand
    int g = 0, item_n = 0, k = 0;
    while (true) {
      bool done = false;
      const Item it = next_item(k++, done);
      if (done) break;
      if (it.kind != 0) continue;
      // The item's query rows for this warp, bf16 -> fp16 (loaded now, stored with the first tile).
      const int qr = quarter * 16 + (lane & 15);
      uint32_t qw[32];
      if (q_warp && qr < Hq) {
        const uint4* src = reinterpret_cast<const uint4*>(p.q + ((int64_t)it.b * Hq + qr) * kHeadDim + (lane >> 4) * 64);
#pragma unroll
        for (int v = 0; v < 8; ++v) {
          const uint4 x = src[v];
          const uint32_t xs[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
          for (int e = 0; e < 4; ++e)
            qw[v * 4 + e] = pack_f16x2(__uint_as_float(xs[e] << 16), __uint_as_float(xs[e] & 0xFFFF0000u));
        }
      } else {
#pragma unroll
        for (int v = 0; v < 32; ++v) qw[v] = 0;
      }
      bool ok = true;
      for (int t = 0; t < it.ntiles && ok; ++t, ++g) {
        const int c = g & 1;
        const int s0 = (2 * g) % NST, s1 = (2 * g + 1) % NST;
        ok = mbar_wait_abortable(&raw_full[s0], ((2 * g) / NST) & 1, abort_flag) &&
             mbar_wait_abortable(&raw_full[s1], ((2 * g + 1) / NST) & 1, abort_flag);
        if (ok && g >= 2) ok = mbar_wait_abortable(&s_full[c], ((g >> 1) - 1) & 1, abort_flag);  // K16[c] free
        if (!ok) break;
        // K: 1024 16-byte units per tile; lanes rotated across chunks (conflict-free).  All loads first.
        {
          uint4 w[kUnits];
          int tts[kUnits], chs[kUnits];
#pragma unroll
          for (int u = 0; u < kUnits; ++u) {
            const int unit = u * (4 * kConvWarps) + (ctid >> 3);
            const int tt = (unit >> 3) * 8 + (ctid & 7);
            const int ch = ((unit & 7) + (ctid & 7)) & 7;
            const int tr = tt & (RT - 1);
            tts[u] = tt;
            chs[u] = ch;
            w[u] = *reinterpret_cast<const uint4*>(raw + (tt < RT ? s0 : s1) * kRawStageBytes + (tr / P) * page_bytes(P) +
                                                   (tr % P) * kHeadDim + ch * 16);
          }
          uint8_t* kd = k16 + c * kOp16Bytes;
#pragma unroll
          for (int u = 0; u < kUnits; ++u) {
            uint32_t a0, a1, a2, a3, a4, a5, a6, a7;
            i8x4_to_f16x4(w[u].x, a0, a1);
            i8x4_to_f16x4(w[u].y, a2, a3);
            i8x4_to_f16x4(w[u].z, a4, a5);
            i8x4_to_f16x4(w[u].w, a6, a7);
            *reinterpret_cast<uint4*>(kd + kmajor_off(tts[u], 2 * chs[u])) = make_uint4(a0, a1, a2, a3);
            *reinterpret_cast<uint4*>(kd + kmajor_off(tts[u], 2 * chs[u] + 1)) = make_uint4(a4, a5, a6, a7);
          }
        }
        // Scales and mask of tile g into slot c: softmax of tile g-2 must be done with the slot.
        if (g >= 2) ok = mbar_wait_abortable(&p_full[c], ((g >> 1) - 1) & 1, abort_flag);
        if (!ok) break;
        if (ctid < T) {
          const int tt = ctid;
          const int s = tt < RT ? s0 : s1;
          const int tr = tt & (RT - 1);
          const int abs_t = (it.tile0 + t) * T + tt;
          const bool valid = abs_t >= it.start && abs_t < it.end && ((page_ok[s] >> (tr / P)) & 1u);
          const float* sc = reinterpret_cast<const float*>(raw + s * kRawStageBytes + (tr / P) * page_bytes(P) +
                                                           2 * P * kHeadDim);
          float* dst = scal + c * 3 * T;
          dst[tt] = valid ? sc[tr % P] * p.scale_log2 : 0.0f;
          dst[T + tt] = valid ? 0.0f : -INFINITY;
          dst[2 * T + tt] = valid ? sc[P + tr % P] : 0.0f;
          if (tt == 0) {
            const int tb = (it.tile0 + t) * T;
            const uint32_t all = (1u << (RT / P)) - 1u;
            tile_full[c] = tb >= it.start && tb + T <= it.end && page_ok[s0] == all && page_ok[s1] == all;
          }
        }
        if (t == 0 && q_warp) {
          // Q[item_n & 1] was last read by the S of an item at least two tiles back: done (K16 wait above).
          tmem_st_16x32bx2_x32<32>(tmem + ((uint32_t)(quarter * 32) << 16) + kColQ + (item_n & 1) * 64, qw);
          tmem_wait_st();
        }
        fence_proxy_async_smem();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&k_full[c]);
        // V: buffer c is free once PV of tile g-2 is done.
        if (g >= 2) ok = mbar_wait_abortable(&v_free[c], ((g >> 1) - 1) & 1, abort_flag);
        if (!ok) break;
        {
          uint4 w[kUnits];
          int tts[kUnits], chs[kUnits];
#pragma unroll
          for (int u = 0; u < kUnits; ++u) {
            const int unit = u * (4 * kConvWarps) + (ctid >> 3);
            const int tt = (unit >> 3) * 8 + (ctid & 7);
            const int ch = ((unit & 7) + (ctid & 7)) & 7;
            const int tr = tt & (RT - 1);
            tts[u] = tt;
            chs[u] = ch;
            w[u] = *reinterpret_cast<const uint4*>(raw + (tt < RT ? s0 : s1) * kRawStageBytes + (tr / P) * page_bytes(P) +
                                                   P * kHeadDim + (tr % P) * kHeadDim + ch * 16);
          }
          uint8_t* vd = v16 + c * kOp16Bytes;
#pragma unroll
          for (int u = 0; u < kUnits; ++u) {
            uint32_t a0, a1, a2, a3, a4, a5, a6, a7;
            i8x4_to_f16x4(w[u].x, a0, a1);
            i8x4_to_f16x4(w[u].y, a2, a3);
            i8x4_to_f16x4(w[u].z, a4, a5);
            i8x4_to_f16x4(w[u].w, a6, a7);
            *reinterpret_cast<uint4*>(vd + mnmajor_off(tts[u], 2 * chs[u])) = make_uint4(a0, a1, a2, a3);
            *reinterpret_cast<uint4*>(vd + mnmajor_off(tts[u], 2 * chs[u] + 1)) = make_uint4(a4, a5, a6, a7);
          }
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(&raw_empty[s0]);
          mbar_arrive(&raw_empty[s1]);
          mbar_arrive(&v_full[c]);
        }
      }
      if (!ok) break;
      ++item_n;
    }
  } else {
    setmaxnreg_inc<kRegsSoft>();
    // ------------------------------------------------------------ softmax + epilogue
    // Two warps per TMEM lane quarter: warp half hf takes tokens [64*hf, 64*hf + 64) of
    // each tile and channels [64*hf, 64*hf + 64) of O; within a warp, thread half th takes
    // 32 of those.  Head row h = 16*quarter + lane%16.  The two warps of a quarter agree
    // on each row's maximum through a small shared exchange and a 64-thread barrier.
    const int sw = warp - kSoftWarp0;
    const int quarter = warp & 3;
    const int hf = sw >> 2;
    const int h = quarter * 16 + (lane & 15);
    const int th = lane >> 4;
    const int tok0 = hf * 64 + th * 32;         // first token (of the tile) this thread handles
    const uint32_t t_lane = (uint32_t)(quarter * 32) << 16;
    const bool warp_live = quarter * 16 < Hq;   // padded rows only: skip the arithmetic
    float* xch = reinterpret_cast<float*>(smem + kOffXch);  // [2][2][64]
    const uint32_t pair_bar = 1 + quarter;      // named barrier of the two warps of this quarter
    int g = 0, item_n = 0, k = 0;
    while (true) {
      bool done = false;
      const Item it = next_item(k++, done);
      if (done) break;
      if (it.kind == 1) {
        // Nothing to attend (L = 0) or an invalid length: out = 0, lse = -inf.
        if (it.invalid && sw == 0 && lane == 0) set_err(p.err, CAI_DEVERR_LENGTH);
        if (h < Hq) {
          float* dst = p.out + ((int64_t)it.b * Hq + h) * kHeadDim + hf * 64 + th * 32;
          for (int d = 0; d < 32; d += 4) *reinterpret_cast<float4*>(dst + d) = make_float4(0.f, 0.f, 0.f, 0.f);
          if (p.lse_out && th == 0 && hf == 0) p.lse_out[(int64_t)it.b * Hq + h] = -INFINITY;
        }
        continue;
      }
      float m_ref = -INFINITY, l_sum = 0.0f;
      bool ok = true;
      for (int t = 0; t < it.ntiles; ++t, ++g) {
        const int c = g & 1;
        ok = mbar_wait_abortable(&s_full[c], (g >> 1) & 1, abort_flag) &&
             mbar_wait_abortable(&k_full[c], (g >> 1) & 1, abort_flag);
        if (!ok) break;
        tc_fence_after();
        const uint32_t scol = kColS + c * 128;
        if (warp_live) {
          uint32_t sr[32];
          tmem_ld_16x32bx2_x32<32>(tmem + t_lane + scol + hf * 64, sr);
          tmem_wait_ld();
          const float* ksc = scal + c * 3 * T + tok0;
          const float* kbias = ksc + T;
          const float* vsc = ksc + 2 * T;
          float mx4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
          if (tile_full[c]) {
#pragma unroll
            for (int j = 0; j < 32; j += 4) {
              const float4 a = *reinterpret_cast<const float4*>(ksc + j);
              const float z0 = __uint_as_float(sr[j]) * a.x, z1 = __uint_as_float(sr[j + 1]) * a.y;
              const float z2 = __uint_as_float(sr[j + 2]) * a.z, z3 = __uint_as_float(sr[j + 3]) * a.w;
              sr[j] = __float_as_uint(z0);
              sr[j + 1] = __float_as_uint(z1);
              sr[j + 2] = __float_as_uint(z2);
              sr[j + 3] = __float_as_uint(z3);
              mx4[0] = fmaxf(mx4[0], z0);
              mx4[1] = fmaxf(mx4[1], z1);
              mx4[2] = fmaxf(mx4[2], z2);
              mx4[3] = fmaxf(mx4[3], z3);
            }
          } else {
#pragma unroll
            for (int j = 0; j < 32; j += 4) {
              const float4 a = *reinterpret_cast<const float4*>(ksc + j);
              const float4 bb = *reinterpret_cast<const float4*>(kbias + j);
              const float z0 = fmaf(__uint_as_float(sr[j]), a.x, bb.x), z1 = fmaf(__uint_as_float(sr[j + 1]), a.y, bb.y);
              const float z2 = fmaf(__uint_as_float(sr[j + 2]), a.z, bb.z), z3 = fmaf(__uint_as_float(sr[j + 3]), a.w, bb.w);
              sr[j] = __float_as_uint(z0);
              sr[j + 1] = __float_as_uint(z1);
              sr[j + 2] = __float_as_uint(z2);
              sr[j + 3] = __float_as_uint(z3);
              mx4[0] = fmaxf(mx4[0], z0);
              mx4[1] = fmaxf(mx4[1], z1);
              mx4[2] = fmaxf(mx4[2], z2);
              mx4[3] = fmaxf(mx4[3], z3);
            }
          }
          float mx = fmaxf(fmaxf(mx4[0], mx4[1]), fmaxf(mx4[2], mx4[3]));
          mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
          // Row maximum over the whole tile: exchange with the other warp of this quarter.
          float* xg = xch + (g & 1) * 128;
          if (th == 0) xg[hf * 64 + h] = mx;
          named_barrier_sync(pair_bar, 64);
          mx = fmaxf(mx, xg[(1 - hf) * 64 + h]);
          const bool raise = mx > m_ref + kRescaleThreshold;
          const float alpha = raise ? ex2_approx(m_ref - mx) : 1.0f;
          if (t > 0 && __any_sync(0xffffffffu, raise)) {
            // O holds earlier tiles of this item: wait for the previous PV, then rescale this warp's half.
            ok = mbar_wait_abortable(&v_free[(g - 1) & 1], ((g - 1) >> 1) & 1, abort_flag);
            if (ok) {
              tc_fence_after();
              uint32_t o[32];
              tmem_ld_16x32bx2_x32<32>(tmem + t_lane + kColO + hf * 64, o);
              tmem_wait_ld();
#pragma unroll
              for (int j = 0; j < 32; ++j) o[j] = __float_as_uint(__uint_as_float(o[j]) * alpha);
              tmem_st_16x32bx2_x32<32>(tmem + t_lane + kColO + hf * 64, o);
              tmem_wait_st();
            }
          }
          if (raise) {
            l_sum *= alpha;
            m_ref = mx;
          }
          const float m_use = m_ref == -INFINITY ? 0.0f : m_ref;
          uint32_t pw[16];
          float l4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
          for (int j = 0; j < 32; j += 4) {
            const float4 vs = *reinterpret_cast<const float4*>(vsc + j);
            const float e0 = ex2_approx(__uint_as_float(sr[j]) - m_use);
            const float e1 = ex2_approx(__uint_as_float(sr[j + 1]) - m_use);
            const float e2 = ex2_approx(__uint_as_float(sr[j + 2]) - m_use);
            const float e3 = ex2_approx(__uint_as_float(sr[j + 3]) - m_use);
            l4[0] += e0;
            l4[1] += e1;
            l4[2] += e2;
            l4[3] += e3;
            pw[j / 2] = pack_f16x2(e0 * vs.x, e1 * vs.y);
            pw[j / 2 + 1] = pack_f16x2(e2 * vs.z, e3 * vs.w);
          }
          l_sum += (l4[0] + l4[1]) + (l4[2] + l4[3]);
          // P (fp16 pairs) over the first 64 columns of the S buffer: tokens 2c, 2c+1 in column c.
          tmem_st_16x32bx2_x16<16>(tmem + t_lane + scol + hf * 32, pw);
          tmem_wait_st();
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&p_full[c]);
        if (!ok) break;
      }
      if (!ok) break;
      // ---- end of item: normalise this thread's 32 channels of its row of O and write them.
      if (!mbar_wait_abortable(o_full, item_n & 1, abort_flag)) break;
      tc_fence_after();
      if (warp_live) {
        // Row sum over the four threads of the row (two lanes here, two in the other warp).
        float l_half = l_sum + __shfl_xor_sync(0xffffffffu, l_sum, 16);
        float* xs = xch + 256;  // [2][64]: the sums, after the two maxima buffers
        if (th == 0) xs[hf * 64 + h] = l_half;
        named_barrier_sync(pair_bar, 64);
        const float l_row = l_half + xs[(1 - hf) * 64 + h];
        named_barrier_sync(pair_bar, 64);  // both have read before the slots are reused
        const float inv = l_row > 0.0f ? 1.0f / l_row : 0.0f;
        uint32_t o[32];
        tmem_ld_16x32bx2_x32<32>(tmem + t_lane + kColO + hf * 64, o);
        tmem_wait_ld();
        if (h < Hq) {
          const int d0 = hf * 64 + th * 32;
          float* dst = it.direct ? p.out + ((int64_t)it.b * Hq + h) * kHeadDim + d0
                                 : p.ws_o + (((int64_t)it.b * p.plan.max_splits + it.split) * Hq + h) * kHeadDim + d0;
#pragma unroll
          for (int j = 0; j < 32; j += 4)
            *reinterpret_cast<float4*>(dst + j) =
                make_float4(__uint_as_float(o[j]) * inv, __uint_as_float(o[j + 1]) * inv,
                            __uint_as_float(o[j + 2]) * inv, __uint_as_float(o[j + 3]) * inv);
          if (th == 0 && hf == 0) {
            const float lse2 = l_row > 0.0f ? m_ref + __log2f(l_row) : -INFINITY;
            if (it.direct) {
              if (p.lse_out) p.lse_out[(int64_t)it.b * Hq + h] = lse2 * kLn2;
            } else {
              p.ws_lse[((int64_t)it.b * p.plan.max_splits + it.split) * Hq + h] = lse2;
            }
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(o_empty);
      ++item_n;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (tid == 0 && *abort_flag) set_err(p.err, CAI_DEVERR_TIMEOUT);
  if (warp == 0) tmem_dealloc(tmem, kTmemCols);
}

// One warp per (sequence, head): merge the partial outputs of the splits by
// their log-sum-exp: out = sum_j 2^(lse_j - M) o_j / sum_j 2^(lse_j - M).
__global__ void __launch_bounds__(128) combine_kernel(const DecodeParams p, int page_size) {
  const int gw = (int)((blockIdx.x * (int64_t)blockDim.x + threadIdx.x) >> 5);
  const int lane = threadIdx.x & 31;
  const int Hq = p.num_heads;
  if (gw >= p.batch * Hq) return;
  const int b = gw / Hq, h = gw - b * Hq;
  const SeqSplits sp = seq_splits(p.ctx_len[b], p.window, p.max_pages * page_size, p.plan.chunk);
  if (!sp.valid || sp.nsplit <= 1) return;  // written by the decode kernel itself
  const int S = p.plan.max_splits;
  const float* lse = p.ws_lse + (int64_t)b * S * Hq + h;
  float M = -INFINITY;
  for (int j = 0; j < sp.nsplit; ++j) M = fmaxf(M, lse[(int64_t)j * Hq]);
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  float wsum = 0.0f;
  if (M != -INFINITY) {
    for (int j = 0; j < sp.nsplit; ++j) {
      const float w = ex2_approx(lse[(int64_t)j * Hq] - M);
      const float4 o = reinterpret_cast<const float4*>(p.ws_o + (((int64_t)b * S + j) * Hq + h) * kHeadDim)[lane];
      acc.x = fmaf(w, o.x, acc.x);
      acc.y = fmaf(w, o.y, acc.y);
      acc.z = fmaf(w, o.z, acc.z);
      acc.w = fmaf(w, o.w, acc.w);
      wsum += w;
    }
  }
  const float inv = wsum > 0.0f ? 1.0f / wsum : 0.0f;
  reinterpret_cast<float4*>(p.out + ((int64_t)b * Hq + h) * kHeadDim)[lane] =
      make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv);
  if (p.lse_out && lane == 0) p.lse_out[(int64_t)b * Hq + h] = wsum > 0.0f ? (M + __log2f(wsum)) * kLn2 : -INFINITY;
}

}  // namespace

int num_sms() {
  static int cached[64] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 64 && cached[dev]) return cached[dev];
  int n = 0;
  cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
  if (n <= 0) n = 1;
  if (dev < 64) cached[dev] = n;
  return n;
}

namespace {

template <int P>
cudaError_t launch_decode_p(const DecodeParams& p, cudaStream_t stream) {
  static bool attr_set[64] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 64 && !attr_set[dev]) {
    // The register split inside the kernel assumes the launch register count.
    cudaFuncAttributes fa;
    cudaError_t e = cudaFuncGetAttributes(&fa, decode_kernel<P>);
    if (e != cudaSuccess) return e;
    if (fa.numRegs != kRegsLaunch) return cudaErrorInvalidDeviceFunction;
    e = cudaFuncSetAttribute(decode_kernel<P>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    if (e != cudaSuccess) return e;
    attr_set[dev] = true;
  }
  const int64_t items = (int64_t)p.batch * p.plan.max_splits;
  const int grid = (int)(items < num_sms() ? items : num_sms());
  decode_kernel<P><<<grid, kThreads, kSmemBytes, stream>>>(p);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess || p.plan.max_splits <= 1) return e;
  const int64_t warps = (int64_t)p.batch * p.num_heads;
  combine_kernel<<<(unsigned)((warps + 3) / 4), 128, 0, stream>>>(p, P);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_decode(const DecodeParams& p, int page_size, cudaStream_t stream) {
  switch (page_size) {
    case 16: return launch_decode_p<16>(p, stream);
    case 32: return launch_decode_p<32>(p, stream);
    case 64: return launch_decode_p<64>(p, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace cai
