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
//  2. attention: a persistent kernel whose work items are 128-row q-tiles of
//     one sequence, a row being one (new token, head) pair.  Each 128-key tile of
//     the copy is in the tcgen05 operand layout already and arrives by one bulk
//     copy; S = Q K^T runs as tcgen05.mma kind::f16 (bf16, M = N = 128, K = 128)
//     into tensor memory; the online softmax (thread = row; two warps per row,
//     each taking one half of the keys with its own reference, sum and O
//     accumulator, merged at the end of the item) forms logit - reference with
//     one FFMA per key (per-key K scale), applies the causal/window mask on
//     boundary tiles only, raises the reference lazily (when a logit exceeds it
//     by 2^8), and writes P (fp16) into tensor memory, where it is the A operand
//     of O_h += P_h V_h (V from shared memory, MN-major).
#include <cuda_fp16.h>

#include <algorithm>

#include "common.cuh"
#include "ptx.cuh"

namespace cai {
namespace {

constexpr int kRows = 128;                 // query rows per q-tile (MMA M)
constexpr int kQT = 1;                     // q-tiles per work item
constexpr int kKeys = 128;                 // keys per tile (MMA N of S, K of PV)
constexpr int kTileBytes = kKeys * kHeadDim * 2;  // 32 KB of 16-bit values
constexpr int kStagesK = 2;                // K tile slots
constexpr int kStagesV = 3;                // V tile slots (with the tile's K scales, which the softmax reads)
constexpr int kPBuf = 2;                   // P buffers in tensor memory (S has one)
constexpr int kOffQ = 0;                                     // Q
// K tiles and V tiles (with the tile's K scales) have separate rings: a K slot is
// free as soon as S = Q K^T of its tile has run, so the next K tiles load ahead of
// the softmax; a V slot (and its scales, which the softmax of its tile reads first)
// is free after its PV, so the V ring is one slot deeper.
constexpr int kOffK = kOffQ + kQT * kRows * kHeadDim * 2;   // K[kStagesK]
constexpr int kVSlotBytes = kTileBytes + kKeys * 4;          // V (scaled), K scales
constexpr int kOffV = kOffK + kStagesK * kTileBytes;         // V[kStagesV]
constexpr int kOffXch = kOffV + kStagesV * kVSlotBytes;      // softmax exchange: row references, row sums [2][128] each
constexpr int kOffBars = kOffXch + 4 * kRows * 4;
// k_full, k_empty [kStagesK]; v_full, v_empty [kStagesV]; q_full; s_full, s_read;
// p_full [2 key halves][kPBuf]; pv_done [kPBuf] (one per P buffer); o_full, o_empty;
// the MMA issuers' last commits.
constexpr int kNumBars = 2 * kStagesK + 2 * kStagesV + 1 + 2 + 3 * kPBuf + 2 + 1;
constexpr int kOffMisc = kOffBars + 8 * kNumBars;
// Varlen dequant: sequences whose tiles one block numbers in shared memory.
constexpr int kMaxCompactSeqs = 8192;
// A varlen call's item list (see PrefillParams::compact): its count, then the dense
// q-tile number of each item, in shared memory that only such a launch asks for.
constexpr int kMaxCompactItems = 4096;
constexpr int kOffTable = kOffMisc + 32;  // after the tmem slot and the wait state (+8)
constexpr int kSmemBytes = kOffTable + 1024;  // without the list; ... and alignment slack
constexpr int kSmemBytesMax = kSmemBytes + (kMaxCompactItems + 4) * 4;
static_assert(kOffXch % 16 == 0 && kOffBars % 8 == 0, "shared-memory layout");
// Warpgroup 0: K/V producer (warp 0), S issuer (warp 1), PV issuer (warp 2), a spare warp;
// warpgroups 1 and 2: the softmax, key half 0 and key half 1 of every row.  The block
// is launched with 168 registers per thread (384 threads; 3 warps x 32 x 168 =
// 16128 of a sub-partition's 16384), then warpgroup 0 shrinks to 72 and the
// softmax groups grow to 216: 128 * (72 + 216 + 216) = 64512 = 384 * 168, so
// the growth is covered exactly by what warpgroup 0 gives back.  The host
// checks the launch register count before the first launch.
constexpr int kThreads = 384;
constexpr int kRegsCtl = 72, kRegsSoft = 216;
constexpr int kRegsLaunch = 168;
static_assert(kRegsCtl * 128 + kRegsSoft * 256 <= kRegsLaunch * kThreads, "register split");
constexpr uint32_t kTmemCols = 512;        // S (128 columns), P[2] (64 each), O[2] (128 each, one per key half)
constexpr float kRescaleThreshold = 8.0f;

struct PrefillParams {
  const uint8_t* pages;
  int32_t num_pages, page_size, max_pages;
  const int32_t* table;
  const int32_t* prefix_len;
  const uint16_t* q;      // bf16 [rows of new tokens][Hq][128], sequence b's rows from q_row0(b)
  const int32_t* q_off;   // [B + 1] packed new-token offsets, or null: sequence b has n_new rows at b * n_new
  int32_t batch, n_new, total_new, num_heads, log2_heads, window, kt_rows, qtiles;  // n_new: the most per sequence; qtiles per sequence
  float scale_log2;
  // Work items: items [0, full_items) are whole q-tiles; the q-tiles after them (the
  // last, partial wave of a persistent grid) are cut into `pieces` key ranges each,
  // item full_items + t being piece t % pieces of q-tile full_items + t / pieces.  A
  // piece writes its normalised partial output and log2-sum-exp to piece_o / piece_lse
  // ([t][128 rows][128] and [t][128]); combine_pieces_kernel merges them.
  int32_t full_items, pieces, num_items;
  uint64_t wait_ns;  // limit of every bounded wait inside the kernel
  int32_t drop_stage;  // fault injection: K tile each CTA skips (-1: none)
  int32_t skip_single;  // see PrefillLaunch
  // Varlen calls: the items are only the q-tiles that hold rows, sequence by sequence,
  // through a list of their dense numbers that every CTA builds at its start (the dense
  // numbering, qtiles slots per sequence for the longest one, would make the grid walk
  // the empty slots of every short or one-token sequence); past kMaxCompactItems real
  // q-tiles, the dense numbering.  No pieces then.
  int32_t compact;
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

// 8 x 8 bytes across the 8 lanes q = lane % 8 of an aligned group: lane q enters with
// row q (bytes 0..3 in a, 4..7 in b) and leaves with column q (rows 0..3 in a, 4..7 in
// b).  Three exchanges: 4-byte blocks with lane q ^ 4, 2-byte blocks with q ^ 2, bytes
// with q ^ 1.
__device__ __forceinline__ void transpose8x8_bytes(uint32_t& a, uint32_t& b, int q) {
  {
    const uint32_t r = __shfl_xor_sync(0xffffffffu, (q & 4) ? a : b, 4);
    if (q & 4) a = r;
    else b = r;
  }
  {
    const uint32_t ra = __shfl_xor_sync(0xffffffffu, a, 2), rb = __shfl_xor_sync(0xffffffffu, b, 2);
    a = (q & 2) ? __byte_perm(ra, a, 0x7632) : __byte_perm(a, ra, 0x5410);
    b = (q & 2) ? __byte_perm(rb, b, 0x7632) : __byte_perm(b, rb, 0x5410);
  }
  {
    const uint32_t ra = __shfl_xor_sync(0xffffffffu, a, 1), rb = __shfl_xor_sync(0xffffffffu, b, 1);
    a = (q & 1) ? __byte_perm(a, ra, 0x3715) : __byte_perm(a, ra, 0x6240);
    b = (q & 1) ? __byte_perm(b, rb, 0x3715) : __byte_perm(b, rb, 0x6240);
  }
}

// Tile `tile` of sequence b's copy, by a block of 256 threads, one warp per 16 rows;
// a tile that no query of the chunk reads returns at once.
__device__ __forceinline__ void dequant_tile(const PrefillParams& p, int b, int tile) {
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
  // Warp w takes keys 16w .. 16w + 15 of the tile in two groups of 8; in each group
  // lane l handles key r0 + (l % 8) and channel chunk 4i + l / 8 (8 channels) for
  // i = 0..3, so that a store instruction writes four whole 128-byte lines of the
  // tiled copy (chunk c of 8 consecutive keys is 128 contiguous bytes).
  const int warp = threadIdx.x >> 5;
  const int P = p.page_size;
  for (int grp = 0; grp < 2; ++grp) {
    const int rr = warp * 16 + grp * 8 + (lane & 7);  // key within the tile
    const int t = tile * kKeys + rr;
    const uint8_t* pg = nullptr;
    int slot = 0;
    float ksc = 0.0f, vsc = 0.0f;
    if (t < len && t >= lo_min) {
      const int32_t page = p.table[(int64_t)b * p.max_pages + t / P];
      if (page >= 0 && page < p.num_pages) {
        slot = t % P;
        pg = p.pages + (int64_t)page * page_bytes(P);
        const float* sc = reinterpret_cast<const float*>(pg + 2 * P * kHeadDim);
        ksc = sc[slot] * p.scale_log2;
        vsc = sc[P + slot];
      } else if (lane < 8 && p.err) {
        atomicOr(p.err, CAI_DEVERR_PAGE);
      }
    }
    // The page of the group's 8 keys (one page: 8 divides P), for the V loads, if any of
    // them is attended.
    const int t0 = tile * kKeys + warp * 16 + grp * 8;
    const uint8_t* pg8 = nullptr;
    if (t0 < len && t0 + 8 > lo_min) {
      const int32_t page = p.table[(int64_t)b * p.max_pages + t0 / P];
      if (page >= 0 && page < p.num_pages) pg8 = p.pages + (int64_t)page * page_bytes(P) + P * kHeadDim + t0 % P;
    }
    const int64_t row = (int64_t)b * p.kt_rows + t;
    if (lane < 8) p.ks[row] = ksc;
    uint16_t* kt = p.kb + ((int64_t)b * p.kt_rows + tile * kKeys) * kHeadDim + rr * 8;
    uint16_t* vt = p.vh + ((int64_t)b * p.kt_rows + tile * kKeys) * kHeadDim + rr * 8;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int c = 4 * i + (lane >> 3);  // channels 8c .. 8c + 7
      uint2 kw = make_uint2(0u, 0u);
      if (pg) kw = *reinterpret_cast<const uint2*>(pg + slot * kHeadDim + c * 8);
      // V is channel-major in the page (channel d's P codes at d * P): lane q of the 8
      // lanes of chunk c loads channel 8c + q of the group's 8 keys (8 contiguous bytes),
      // and the transpose leaves each lane the 8 channels of its own key.
      uint32_t vw[2] = {0u, 0u};
      if (pg8) {
        const uint2 v8 = *reinterpret_cast<const uint2*>(pg8 + (c * 8 + (lane & 7)) * P);
        vw[0] = v8.x;
        vw[1] = v8.y;
      }
      transpose8x8_bytes(vw[0], vw[1], lane & 7);
      if (!pg) vw[0] = vw[1] = 0u;
      // int8 -> bf16 (K) and int8 -> fp16 (V): exact for |code| <= 127.
      uint32_t ko[4], vo[4];
#pragma unroll
      for (int e = 0; e < 8; e += 2) {
        const uint32_t kx = e < 4 ? kw.x : kw.y, vx = vw[e >> 2];
        const float k0 = (float)(int8_t)(kx >> (8 * (e & 3))), k1 = (float)(int8_t)(kx >> (8 * ((e & 3) + 1)));
        ko[e / 2] = (__float_as_uint(k0) >> 16) | (__float_as_uint(k1) & 0xFFFF0000u);  // small integers: exact
        const float v0 = (float)(int8_t)(vx >> (8 * (e & 3))), v1 = (float)(int8_t)(vx >> (8 * ((e & 3) + 1)));
        const __half2 hv = __floats2half2_rn(v0 * vsc, v1 * vsc);  // V scale applied here: P needs no per-key factor
        vo[e / 2] = *reinterpret_cast<const uint32_t*>(&hv);
      }
      *reinterpret_cast<uint4*>(kt + c * 1024) = make_uint4(ko[0], ko[1], ko[2], ko[3]);
      *reinterpret_cast<uint4*>(vt + c * 1024) = make_uint4(vo[0], vo[1], vo[2], vo[3]);
    }
  }
}

// Tiles of sequence b's copy that the dequant pass writes: [*lo, *lo + count).  A sequence
// whose lengths are invalid writes none (and is flagged).
__device__ __forceinline__ int dequant_tiles(const PrefillParams& p, int b, int* lo) {
  const int32_t p0 = p.prefix_len[b];
  const SeqRows sr = seq_rows(p, b);
  *lo = 0;
  if (!seq_ok(p, p0, sr.n)) {
    if (p.err) atomicOr(p.err, CAI_DEVERR_LENGTH);
    return 0;
  }
  if (sr.n == 0) return 0;
  const int len = p0 + sr.n;
  const int lo_min = p.window > 0 ? max(0, p0 + 1 - p.window) : 0;
  *lo = lo_min / kKeys;
  return (len + kKeys - 1) / kKeys - *lo;
}

// One block per 128-key tile of a sequence (blockIdx.y = sequence).
__global__ void __launch_bounds__(256) dequant_kernel(const PrefillParams p) {
  dequant_tile(p, blockIdx.y, blockIdx.x);
}

// Varlen calls: a grid-stride loop over only the tiles some query reads.  Each block
// first numbers them (a block-wide scan of every sequence's tile count into dynamic
// shared memory, first[b] = number of sequence b's first tile, first[batch] = total);
// the dense grid of the chunk calls would launch a block for every tile slot of every
// sequence, most of them idle for the one-token rows of a mixed batch.
__global__ void __launch_bounds__(256) dequant_compact_kernel(const PrefillParams p) {
  extern __shared__ int32_t first[];
  __shared__ int32_t warp_sum[8];
  const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
  const int B = p.batch;
  const int per = (B + 255) / 256;
  const int b0 = min(B, t * per), b1 = min(B, b0 + per);
  int sum = 0, lo;
  for (int b = b0; b < b1; ++b) sum += dequant_tiles(p, b, &lo);
  int incl = sum;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int v = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += v;
  }
  if (lane == 31) warp_sum[warp] = incl;
  __syncthreads();
  int before = 0;
  for (int w = 0; w < warp; ++w) before += warp_sum[w];
  int run = before + incl - sum;
  for (int b = b0; b < b1; ++b) {
    first[b] = run;
    run += dequant_tiles(p, b, &lo);
  }
  if (t == 255) first[B] = before + incl;
  __syncthreads();
  const int total = first[B];
  for (int w = blockIdx.x; w < total; w += gridDim.x) {
    int l = 0, h = B - 1;  // the last sequence whose first tile is <= w
    while (l < h) {
      const int mid = (l + h + 1) >> 1;
      if (first[mid] <= w) l = mid;
      else h = mid - 1;
    }
    dequant_tiles(p, l, &lo);
    dequant_tile(p, l, lo + (w - first[l]));
  }
}

// One work item: a q-tile (128 consecutive (token, head) rows) of one
// sequence.  ok = false: no MMA work; the softmax groups then write zeros to the
// item's rows below `rows` (an invalid sequence) or nothing (rows beyond the chunk).
struct PItem {
  int b, row0, kt0, nkt;
  int64_t qrow0;  // first packed new-token row of the sequence
  int rows;       // (token, head) rows of the sequence, 0 if its offsets are invalid
  bool ok;
  int piece;      // -1: the whole key range; otherwise the piece's slot in piece_o / piece_lse
};

// q-tiles holding rows of sequence b (0 when it has no rows in this call).
__device__ __forceinline__ int seq_qtiles(const PrefillParams& p, int b) {
  const SeqRows sr = seq_rows(p, b);
  return sr.n > 0 ? (int)(((int64_t)sr.n * p.num_heads + kRows - 1) / kRows) : 0;
}

// The work split of a persistent grid over `total` q-tiles: items [0, full) are whole
// q-tiles; the q-tiles of a partial last wave are cut into `pieces` key ranges so that
// wave ends sooner (with r q-tiles left over, pieces = grid / r, at most 4), item
// full + t being piece t % pieces of q-tile full + t / pieces; num items in all.  The
// host applies it to a chunk call's q-tiles.
struct WorkSplit {
  int full, pieces, num;
};
__host__ __device__ inline WorkSplit work_split(int64_t total, int grid) {
  const int64_t rem = grid > 0 ? total % grid : 0;
  int pieces = rem > 0 ? (int)(grid / rem) : 1;
  if (pieces > 4) pieces = 4;
  if (pieces < 2) pieces = 1;
  WorkSplit w;
  w.pieces = pieces;
  w.full = (int)(pieces > 1 ? total - rem : total);
  w.num = (int)(w.full + (pieces > 1 ? rem * pieces : 0));
  return w;
}

// list: a varlen call's q-tile numbers (entry i for q-tile i - list_first), or null.
__device__ __forceinline__ PItem prefill_item(const PrefillParams& p, int idx, const int32_t* list,
                                              const WorkSplit& ws, int list_first = 0) {
  PItem it;
  int qti = idx, piece = -1;
  if (idx >= ws.full) {
    const int t = idx - ws.full;
    qti = ws.full + t / ws.pieces;
    piece = t % ws.pieces;
    it.piece = t;
  } else {
    it.piece = -1;
  }
  const int qt = list ? list[qti - list_first] : qti;
  it.b = qt / p.qtiles;
  it.row0 = (qt - it.b * p.qtiles) * (kQT * kRows);
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
  if (piece >= 0) {  // key tiles [per * piece, per * (piece + 1)) of the q-tile's range
    const int per = (it.nkt + ws.pieces - 1) / ws.pieces;
    const int a = min(it.nkt, per * piece), e = min(it.nkt, per * (piece + 1));
    it.kt0 += a;
    it.nkt = e - a;
  }
  return it;
}

// Operand tiles in shared memory: element (r, k) of a 128x128 16-bit tile at
// (k/8)*2048 + r*16 + (k%8)*2 -- the order in which the dequant pass writes each
// tile of its copy, so one bulk copy lands it.  As a K-major operand: LBO = 2048
// (next 8 k), SBO = 128 (next 8 rows).  As an MN-major operand (rows = K, k = N):
// LBO = 128, SBO = 2048.
//
// Persistent CTAs, one per SM, each taking q-tiles in turn.  Roles: warp 0 loads
// K/V tiles (one bulk copy each) into 2-slot K and V rings; warp 1 issues
// S(g) = Q K(g)^T into the one S buffer as soon as K(g) is loaded and the softmax
// has read S(g - 1) into registers, so S of the next tile runs during this tile's
// exponentials; warp 2 issues O_h += P_h(g) V_h(g) for both key halves h, P from
// two alternating buffers; warps 4-7 and 8-11 run the softmax of key half 0 and
// key half 1 of every row (thread = row, 64 keys per tile each), each half with
// its own reference, sum and accumulator, and merge the halves into the outputs at
// the end of the item (channel half each).
// kCompact: a varlen call's launch (p.compact): its items go through the item list.
// Chunk calls compile without that path (its one branch per item cost them 2%).
template <bool kCompact>
__global__ void __launch_bounds__(kThreads, 1) prefill_kernel(const PrefillParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kOffBars);
  uint64_t* k_full = bars;                     // [kStagesK] producer -> S issuer (tx bytes)
  uint64_t* k_empty = k_full + kStagesK;       // [kStagesK] S issuer commit after S of the tile
  uint64_t* v_full = k_empty + kStagesK;       // [kStagesV] producer -> PV issuer, softmax (V and K scales)
  uint64_t* v_empty = v_full + kStagesV;       // [kStagesV] PV issuer commit after PV of the tile
  uint64_t* q_full = v_empty + kStagesV;       // softmax -> S issuer (8 warps)
  uint64_t* s_full = q_full + 1;               // S issuer commit after S
  uint64_t* s_read = s_full + 1;               // softmax -> S issuer (8 warps): S read, the next may overwrite it
  uint64_t* p_full = s_read + 1;               // [2][kPBuf] softmax half h -> PV issuer (4 warps): P in buffer b
  uint64_t* pv_done = p_full + 2 * kPBuf;      // [kPBuf] PV issuer commit after both PVs reading P buffer b
  uint64_t* o_full = pv_done + kPBuf;          // PV issuer commit after an item's last PVs
  uint64_t* o_empty = o_full + 1;              // softmax -> PV issuer after reading O (8 warps)
  uint64_t* mma_drain = o_empty + 1;           // the MMA issuers' last commits, at exit
  float* xref = reinterpret_cast<float*>(smem + kOffXch);  // [2 halves][128 rows] half-row references
  float* xsum = xref + 2 * kRows;                          // [2 halves][128 rows] half-row sums
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kOffMisc);
  volatile WaitState* const wctl = reinterpret_cast<volatile WaitState*>(smem + kOffMisc + 8);
  volatile int32_t* abort_flag = &wctl->abort;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int Hq = p.num_heads;
  constexpr uint32_t kColP = 128;  // P buffer b at kColP + b * 64 (key half h in its 32 columns at + h * 32); S at 0
  constexpr uint32_t kColO = 256;  // O of key half h at kColO + h * 128
  constexpr uint32_t kSoftBar = 1;
  constexpr uint32_t kSoftThreads = 256;

  if (warp == 0) tmem_alloc(tmem_slot, kTmemCols);
  if (tid == 0) {
    for (int s = 0; s < kStagesK; ++s) {
      mbar_init(&k_full[s], 1);
      mbar_init(&k_empty[s], 1);
    }
    for (int s = 0; s < kStagesV; ++s) {
      mbar_init(&v_full[s], 1);
      mbar_init(&v_empty[s], 1);
    }
    mbar_init(q_full, 8);
    mbar_init(s_full, 1);
    mbar_init(s_read, 8);
    for (int b = 0; b < kPBuf; ++b) {
      mbar_init(&p_full[b], 4);
      mbar_init(&p_full[kPBuf + b], 4);
      mbar_init(&pv_done[b], 1);
    }
    mbar_init(o_full, 1);
    mbar_init(o_empty, 8);
    mbar_init(mma_drain, 2);
    *abort_flag = 0;
    wctl->limit_ns = p.wait_ns;
    fence_barrier_init();
  }
  if (kCompact && warp == 3) {
    // The item list: lane l sums the q-tiles of a run of sequences, a warp scan gives
    // each run its first item, and each lane writes its run's items; the count is -1
    // (the dense numbering) when they do not fit.
    int32_t* hdr = reinterpret_cast<int32_t*>(smem + kOffTable);
    int32_t* list = hdr + 4;
    const int per = (p.batch + 31) / 32;
    const int b0 = min(p.batch, lane * per), b1 = min(p.batch, b0 + per);
    int sum = 0;
    for (int b = b0; b < b1; ++b) sum += seq_qtiles(p, b);
    int incl = sum;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += v;
    }
    const int total = __shfl_sync(0xffffffffu, incl, 31);
    if (total <= kMaxCompactItems) {
      int run = incl - sum;
      for (int b = b0; b < b1; ++b) {
        const int n = seq_qtiles(p, b);
        for (int j = 0; j < n; ++j) list[run + j] = b * p.qtiles + j;
        run += n;
      }
    }
    if (lane == 0) *hdr = total <= kMaxCompactItems ? total : -1;
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  // A varlen call's decode launch, next in the stream, shares no memory with this grid:
  // it may start now, its CTAs taking the SMs that this grid's CTAs leave.  (Chunk calls
  // do not trigger early: measured 3.6% slower on the append-prefill workload.)
  if (kCompact) grid_launch_dependents();
  // A varlen call's item list, if it was built (above).
  const int n_list = kCompact ? *reinterpret_cast<const int32_t*>(smem + kOffTable) : -1;
  const int32_t* table = n_list >= 0 ? reinterpret_cast<const int32_t*>(smem + kOffTable + 16) : nullptr;
  // A varlen call's q-tiles are whole (pieces measured no faster there): the host gives it
  // full_items = num_items = the dense count, which no listed item reaches.
  WorkSplit ws;
  ws.full = p.full_items;
  ws.pieces = p.pieces;
  ws.num = n_list >= 0 ? n_list : p.num_items;
  const int num_items = ws.num;

  if (warp < 4) {
   setmaxnreg_dec<kRegsCtl>();
   if (warp == 0) {
    // ------------------------------------------------------------ K/V producer
    if (lane == 0) {
      int g = 0, gk = 0, gv = 0;  // tiles; tiles whose K and V loads were issued (or dropped)
      for (int idx = blockIdx.x; idx < num_items && !*abort_flag; idx += gridDim.x) {
        const PItem it = prefill_item(p, idx, table, ws);
        const int64_t seq_row0 = (int64_t)it.b * p.kt_rows;
        for (int j = 0; j < it.nkt; ++j, ++g) {
          const int sk = g % kStagesK, sv = g % kStagesV;
          const int64_t row = seq_row0 + (int64_t)(it.kt0 + j) * kKeys;
          if (g >= kStagesK && !mbar_wait_polled(&k_empty[sk], ((g / kStagesK) - 1) & 1, wctl)) break;
          if (g != p.drop_stage) {  // (fault injection: that K tile is never loaded)
            mbar_arrive_expect_tx(&k_full[sk], kTileBytes);
            bulk_g2s(smem + kOffK + sk * kTileBytes, p.kb + row * kHeadDim, kTileBytes, &k_full[sk]);
          }
          gk = g + 1;
          if (g >= kStagesV && !mbar_wait_polled(&v_empty[sv], ((g / kStagesV) - 1) & 1, wctl)) break;
          uint8_t* vs = smem + kOffV + sv * kVSlotBytes;
          mbar_arrive_expect_tx(&v_full[sv], kVSlotBytes);
          bulk_g2s(vs, p.vh + row * kHeadDim, kTileBytes, &v_full[sv]);
          bulk_g2s(vs + kTileBytes, p.ks + row, kKeys * 4, &v_full[sv]);
          gv = g + 1;
        }
      }
      // Every slot this producer armed has landed before the CTA goes away, whatever
      // happened to the other roles (copies into a CTA's shared memory must not outlive it).
      for (int i = gk > kStagesK ? gk - kStagesK : 0; i < gk; ++i)
        if (i != p.drop_stage) mbar_wait_drain(&k_full[i % kStagesK], (i / kStagesK) & 1);
      for (int i = gv > kStagesV ? gv - kStagesV : 0; i < gv; ++i) mbar_wait_drain(&v_full[i % kStagesV], (i / kStagesV) & 1);
    }
   } else if (warp == 1 || warp == 2) {
    // ------------------------------------------------------------ MMA issuers
    // Warp 1 issues S = Q K^T, warp 2 issues O += P V: one thread issues a
    // 128 x 128 x 16 MMA only about every 115 cycles (measured; the tensor core takes
    // about 64), so the two streams go out from two threads.  S(g) overwrites S once
    // the softmax has read S(g - 1) into registers, so it runs during that softmax's
    // exponentials; P has buffers of its own.
    if (lane == 0) {
      constexpr uint32_t idesc_s = idesc_bf16_f32(kRows, kKeys, 0, 0);
      constexpr uint32_t idesc_o = idesc_f16_f32(kRows, kHeadDim, 0, 1);
      const bool s_issuer = warp == 1;
      // Descriptor bases; a K step adds 4096 bytes (S operands) or 256 bytes (V),
      // i.e. 256 or 16 to the address field (shared addresses stay below 2^18).
      const uint64_t dq = smem_desc(smem_addr(smem + kOffQ), 2048, 128);
      const uint64_t dk0 = smem_desc(smem_addr(smem + kOffK), 2048, 128);
      const uint64_t dv0 = smem_desc(smem_addr(smem + kOffV), 128, 2048);
      int g = 0, n = 0;
      bool ok = true;
      for (int idx = blockIdx.x; idx < num_items && ok && !*abort_flag; idx += gridDim.x) {
        const PItem it = prefill_item(p, idx, table, ws);
        if (!it.ok || it.nkt == 0) continue;  // no MMA work; the softmax writes its zeros
        if (s_issuer) ok = mbar_wait_polled(q_full, n & 1, wctl);
        for (int j = 0; j < it.nkt && ok; ++j, ++g) {
          const int sk = g % kStagesK, sv = g % kStagesV, b = g % kPBuf;
          if (s_issuer) {
            ok = mbar_wait_polled(&k_full[sk], (g / kStagesK) & 1, wctl) &&
                 (g == 0 || mbar_wait_polled(s_read, (g - 1) & 1, wctl));
            if (!ok) break;
            tc_fence_after();
            const uint64_t dk = dk0 + (uint64_t)(sk * (kTileBytes / 16));
#pragma unroll
            for (int ks = 0; ks < kHeadDim / 16; ++ks)
              mma_f16_ss(tmem, dq + (uint64_t)(ks * 256), dk + (uint64_t)(ks * 256), idesc_s, ks > 0);
            mma_commit(s_full);
            mma_commit(&k_empty[sk]);
          } else {
            ok = (j > 0 || n == 0 || mbar_wait_polled(o_empty, (n - 1) & 1, wctl)) &&
                 mbar_wait_polled(&v_full[sv], (g / kStagesV) & 1, wctl);
            const uint64_t dv = dv0 + (uint64_t)(sv * (kVSlotBytes / 16));
            // Key half h: O_h += P_h V_h, P_h in its 32 columns of P buffer b.
            for (int hh = 0; hh < 2 && ok; ++hh) {
              ok = mbar_wait_polled(&p_full[hh * kPBuf + b], (g / kPBuf) & 1, wctl);
              if (!ok) break;
              tc_fence_after();
#pragma unroll
              for (int ks = 0; ks < 4; ++ks)
                mma_f16_ts(tmem + kColO + hh * 128, tmem + kColP + b * 64 + hh * 32 + ks * 8,
                           dv + (uint64_t)((hh * 4 + ks) * 16), idesc_o, (j > 0 || ks > 0) ? 1u : 0u);
            }
            if (!ok) break;
            mma_commit(&pv_done[b]);
            mma_commit(&v_empty[sv]);
            if (j == it.nkt - 1) mma_commit(o_full);
          }
        }
        ++n;
      }
      // This issuer's MMAs have completed before tensor memory is freed.
      mma_commit(mma_drain);
      mbar_wait_drain(mma_drain, 0);
    }
   }
  } else {
    setmaxnreg_inc<kRegsSoft>();
    // ------------------------------------------------------------ softmax
    const int h = (warp - 4) >> 2;          // key half of every tile, channel half of the output
    const int quarter = warp & 3;           // TMEM lane quarter
    const int r = quarter * 32 + lane;      // row within the q-tile
    const uint32_t t_lane = (uint32_t)(quarter * 32) << 16;
    uint8_t* qs = smem + kOffQ;
    // The two key halves of a row are independent within an item (own reference, own
    // sum, own O accumulator), so a warp meets no other warp inside the tile loop and
    // decides alone (its waits agree in all lanes).  The 8 warps meet once per item,
    // at its start and to merge the halves; there they stop together if any gave up.
    int g = 0, n = 0;
    bool ok = true;
    for (int idx = blockIdx.x; idx < num_items; idx += gridDim.x) {
      if (bar_red_or(kSoftBar, kSoftThreads, !ok || *abort_flag != 0)) break;
      const PItem it = prefill_item(p, idx, table, ws);
      const int64_t row = it.row0 + r;  // (token, head) row within the sequence
      const bool my_row = row < it.rows;
      const int my_i = (int)(row >> p.log2_heads), my_h = (int)(row & (Hq - 1));
      float* out_row = p.out + ((it.qrow0 + my_i) * Hq + my_h) * kHeadDim + h * 64;
      if (!it.ok) {  // invalid sequence (flagged by the dequant pass): 0 / -inf; beyond the chunk: nothing
        if (my_row) {
          for (int d = 0; d < 64; d += 4) *reinterpret_cast<float4*>(out_row + d) = make_float4(0.f, 0.f, 0.f, 0.f);
          if (h == 0 && p.lse_out) p.lse_out[(it.qrow0 + my_i) * Hq + my_h] = -INFINITY;
        }
        continue;  // no MMA work for this item
      }
      // A piece's partial output row (normalised) and log2-sum-exp, for the merge.
      float* part_row = it.piece >= 0 ? p.piece_o + ((int64_t)it.piece * kRows + r) * kHeadDim + h * 64 : nullptr;
      float* part_lse = it.piece >= 0 ? p.piece_lse + (int64_t)it.piece * kRows + r : nullptr;
      if (it.nkt == 0) {  // a piece with no key tiles (no MMA work): weight zero in the merge
        for (int d = 0; d < 64; d += 4) *reinterpret_cast<float4*>(part_row + d) = make_float4(0.f, 0.f, 0.f, 0.f);
        if (h == 0) *part_lse = -INFINITY;
        continue;
      }
      // This row's query (bf16), zero beyond the chunk: each half writes 8 of its 16 chunks.
      {
        const uint4* src = reinterpret_cast<const uint4*>(p.q + (it.qrow0 * Hq + row) * kHeadDim);
#pragma unroll
        for (int c = 0; c < 8; ++c)
          *reinterpret_cast<uint4*>(qs + (h * 8 + c) * 2048 + r * 16) = my_row ? src[h * 8 + c] : make_uint4(0, 0, 0, 0);
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(q_full);
      const int32_t p0 = p.prefix_len[it.b];
      const int q_pos = p0 + my_i;
      const int k_lo = p.window > 0 ? max(0, q_pos + 1 - p.window) : 0;
      float m_ref = -INFINITY, l_sum = 0.0f;
      for (int j = 0; j < it.nkt; ++j, ++g) {
        const int sv = g % kStagesV, b = g % kPBuf;
        ok = mbar_wait_polled_warp(s_full, g & 1, wctl) &&
             mbar_wait_polled_warp(&v_full[sv], (g / kStagesV) & 1, wctl);
        if (!ok) break;
        tc_fence_after();
        const float* kscale = reinterpret_cast<const float*>(smem + kOffV + sv * kVSlotBytes + kTileBytes) + h * 64;
        const int key0 = (it.kt0 + j) * kKeys + h * 64;
        // z = logit (log2 units) minus this half-row's reference, one FFMA per key.
        const float m_use = m_ref == -INFINITY ? 0.0f : m_ref;
        float z[64];
        {
          uint32_t r0[32], r1[32];
          tmem_ld_32x32b_x32(tmem + t_lane + h * 64, r0);
          tmem_ld_32x32b_x32(tmem + t_lane + h * 64 + 32, r1);
          tmem_wait_ld();
          // S is read: S of the next tile may overwrite it.
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(s_read);
          // Chunk calls: packed fp32 pairs, two FFMAs per instruction (in the varlen
          // instantiation the pairs cost register spills, so it keeps scalar FFMAs).
          const uint64_t nm2 = f2(-m_use, -m_use);
#pragma unroll
          for (int e = 0; e < 32; e += 4) {
            const float4 a = *reinterpret_cast<const float4*>(kscale + e);
            const float4 a2 = *reinterpret_cast<const float4*>(kscale + 32 + e);
            if constexpr (!kCompact) {
              f2_split(f2_fma(f2(__uint_as_float(r0[e]), __uint_as_float(r0[e + 1])), f2(a.x, a.y), nm2), z[e],
                       z[e + 1]);
              f2_split(f2_fma(f2(__uint_as_float(r0[e + 2]), __uint_as_float(r0[e + 3])), f2(a.z, a.w), nm2),
                       z[e + 2], z[e + 3]);
              f2_split(f2_fma(f2(__uint_as_float(r1[e]), __uint_as_float(r1[e + 1])), f2(a2.x, a2.y), nm2),
                       z[32 + e], z[32 + e + 1]);
              f2_split(f2_fma(f2(__uint_as_float(r1[e + 2]), __uint_as_float(r1[e + 3])), f2(a2.z, a2.w), nm2),
                       z[32 + e + 2], z[32 + e + 3]);
            } else {
              z[e] = fmaf(__uint_as_float(r0[e]), a.x, -m_use);
              z[e + 1] = fmaf(__uint_as_float(r0[e + 1]), a.y, -m_use);
              z[e + 2] = fmaf(__uint_as_float(r0[e + 2]), a.z, -m_use);
              z[e + 3] = fmaf(__uint_as_float(r0[e + 3]), a.w, -m_use);
              z[32 + e] = fmaf(__uint_as_float(r1[e]), a2.x, -m_use);
              z[32 + e + 1] = fmaf(__uint_as_float(r1[e + 1]), a2.y, -m_use);
              z[32 + e + 2] = fmaf(__uint_as_float(r1[e + 2]), a2.z, -m_use);
              z[32 + e + 3] = fmaf(__uint_as_float(r1[e + 3]), a2.w, -m_use);
            }
          }
        }
        if (!(key0 >= k_lo && key0 + 63 <= q_pos)) {
#pragma unroll
          for (int c = 0; c < 64; ++c) {
            const int key = key0 + c;
            if (key < k_lo || key > q_pos) z[c] = -INFINITY;
          }
        }
        float mx4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
        for (int c = 0; c < 64; c += 8) {
          mx4[0] = fmax3(mx4[0], z[c], z[c + 1]);
          mx4[1] = fmax3(mx4[1], z[c + 2], z[c + 3]);
          mx4[2] = fmax3(mx4[2], z[c + 4], z[c + 5]);
          mx4[3] = fmax3(mx4[3], z[c + 6], z[c + 7]);
        }
        const float mx = fmaxf(fmaxf(mx4[0], mx4[1]), fmaxf(mx4[2], mx4[3]));
        // Raise the reference when the half-row has none yet, or a logit exceeds it by 2^8.
        const bool raise = m_ref == -INFINITY ? mx > -INFINITY : mx > kRescaleThreshold;
        const float alpha = raise ? ex2_approx(m_ref - (m_use + mx)) : 1.0f;  // 0 when there was no reference
        if (j > 0 && __any_sync(0xffffffffu, raise)) {
          // O_h holds earlier tiles: wait for their PVs, then rescale this row of it.
          ok = mbar_wait_polled_warp(&pv_done[(g - 1) % kPBuf], ((g - 1) / kPBuf) & 1, wctl);
          if (!ok) break;
          tc_fence_after();
#pragma unroll
          for (int c = 0; c < kHeadDim; c += 32) {
            uint32_t o[32];
            tmem_ld_32x32b_x32(tmem + t_lane + kColO + h * 128 + c, o);
            tmem_wait_ld();
#pragma unroll
            for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
            tmem_st_32x32b_x32(tmem + t_lane + kColO + h * 128 + c, o);
          }
          tmem_wait_st();
        }
        if (raise) {
          l_sum *= alpha;
          m_ref = m_use + mx;
#pragma unroll
          for (int c = 0; c < 64; ++c) z[c] -= mx;
        }
        // P = 2^z as fp16 into this half's 32 columns of P buffer b, the A operand of
        // this half's PV, once the PVs of tile g - 2 have read that buffer.
        float l4[4] = {0.f, 0.f, 0.f, 0.f};  // four running sums (chunk calls: as two fp32 pairs)
        uint64_t l01 = 0ull, l23 = 0ull;
        uint32_t pw[32];
#pragma unroll
        for (int e = 0; e < 64; e += 4) {
          const float e0 = ex2_approx(z[e]), e1 = ex2_approx(z[e + 1]);
          const float e2 = ex2_approx(z[e + 2]), e3 = ex2_approx(z[e + 3]);
          if constexpr (!kCompact) {
            l01 = f2_add(l01, f2(e0, e1));
            l23 = f2_add(l23, f2(e2, e3));
          } else {
            l4[0] += e0;
            l4[1] += e1;
            l4[2] += e2;
            l4[3] += e3;
          }
          pw[e / 2] = pack_f16x2(e0, e1);
          pw[e / 2 + 1] = pack_f16x2(e2, e3);
        }
        if constexpr (!kCompact) {
          f2_split(l01, l4[0], l4[1]);
          f2_split(l23, l4[2], l4[3]);
        }
        if (g >= kPBuf) {
          ok = mbar_wait_polled_warp(&pv_done[b], ((g / kPBuf) - 1) & 1, wctl);
          if (!ok) break;
        }
        tmem_st_32x32b_x32(tmem + t_lane + kColP + b * 64 + h * 32, pw);
        l_sum += (l4[0] + l4[1]) + (l4[2] + l4[3]);
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&p_full[h * kPBuf + b]);
      }
      // ---- end of item: merge the halves, O = (w0 O_0 + w1 O_1) / (w0 l_0 + w1 l_1)
      // with w_h = 2^(m_h - M), M the larger reference; this thread writes its channel half.
      xref[h * kRows + r] = m_ref;
      xsum[h * kRows + r] = l_sum;
      if (bar_red_or(kSoftBar, kSoftThreads, !ok)) break;
      const float m0 = xref[r], m1 = xref[kRows + r];
      const float M = fmaxf(m0, m1);
      const float w0 = m0 == -INFINITY ? 0.0f : ex2_approx(m0 - M);
      const float w1 = m1 == -INFINITY ? 0.0f : ex2_approx(m1 - M);
      const float Ls = w0 * xsum[r] + w1 * xsum[kRows + r];
      ok = mbar_wait_polled_warp(o_full, n & 1, wctl);
      if (ok) {
        tc_fence_after();
        const float inv = Ls > 0.0f ? 1.0f / Ls : 0.0f;
        const float c0 = w0 * inv, c1 = w1 * inv;
        float* dst = part_row ? part_row : out_row;
#pragma unroll
        for (int c = 0; c < 64; c += 32) {
          uint32_t o0[32], o1[32];
          tmem_ld_32x32b_x32(tmem + t_lane + kColO + h * 64 + c, o0);
          tmem_ld_32x32b_x32(tmem + t_lane + kColO + 128 + h * 64 + c, o1);
          tmem_wait_ld();
          if (my_row) {
#pragma unroll
            for (int e = 0; e < 32; e += 4)
              *reinterpret_cast<float4*>(dst + c + e) = make_float4(
                  fmaf(c0, __uint_as_float(o0[e]), c1 * __uint_as_float(o1[e])),
                  fmaf(c0, __uint_as_float(o0[e + 1]), c1 * __uint_as_float(o1[e + 1])),
                  fmaf(c0, __uint_as_float(o0[e + 2]), c1 * __uint_as_float(o1[e + 2])),
                  fmaf(c0, __uint_as_float(o0[e + 3]), c1 * __uint_as_float(o1[e + 3])));
          }
        }
        if (h == 0 && my_row) {
          const float lse2 = Ls > 0.0f ? M + __log2f(Ls) : -INFINITY;
          if (part_lse) *part_lse = lse2;
          else if (p.lse_out) p.lse_out[(it.qrow0 + my_i) * Hq + my_h] = lse2 * kLn2;
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(o_empty);
      }
      ++n;
    }
  }
  tc_fence_before();
  __syncthreads();
  if (tid == 0 && *abort_flag && p.err) atomicOr(p.err, CAI_DEVERR_TIMEOUT);
  if (warp == 0) tmem_dealloc(tmem, kTmemCols);
}

// One warp per (split q-tile, row): merge the q-tile's pieces by their log-sum-exp,
// out = sum_j 2^(lse_j - M) o_j / sum_j 2^(lse_j - M), into the row's output.
__global__ void __launch_bounds__(256) combine_pieces_kernel(const PrefillParams p) {
  grid_dependency_wait();
  grid_launch_dependents();
  const int64_t w = (blockIdx.x * (int64_t)blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  WorkSplit ws;
  ws.full = p.full_items;
  ws.pieces = p.pieces;
  ws.num = p.num_items;
  const int split_tiles = (ws.num - ws.full) / ws.pieces;
  if (w >= (int64_t)split_tiles * (kQT * kRows)) return;
  const int sp = (int)(w / (kQT * kRows)), r = (int)(w % (kQT * kRows));
  const PItem it = prefill_item(p, ws.full + sp * ws.pieces, nullptr, ws);
  const int64_t row = it.row0 + r;
  if (!it.ok || row >= it.rows) return;  // invalid sequence (its rows hold zeros) or past the chunk
  const int Hq = p.num_heads;
  const int my_i = (int)(row >> p.log2_heads), my_h = (int)(row & (Hq - 1));
  const int64_t t0 = (int64_t)sp * ws.pieces;
  const float lj = lane < ws.pieces ? p.piece_lse[(t0 + lane) * (kQT * kRows) + r] : -INFINITY;
  float M = lj;
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
  const float wj = (M == -INFINITY || lane >= ws.pieces) ? 0.0f : ex2_approx(lj - M);
  float wsum = wj;
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) wsum += __shfl_xor_sync(0xffffffffu, wsum, o);
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int j = 0; j < ws.pieces; ++j) {
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

}  // namespace

// Partial outputs of the split last wave: at most one piece per CTA of the grid.  The
// region is twice that: a varlen call's decode launch keeps its split partials there
// (fewer splits when they would not fit), and half the room had cost it half its splits.
static int64_t piece_bytes() { return (int64_t)num_sms() * 2 * (kQT * kRows) * (kHeadDim + 1) * 4; }

size_t prefill_workspace_bytes(int32_t batch, int32_t max_pages_per_seq, int32_t page_size) {
  const int64_t kt = ((int64_t)max_pages_per_seq * page_size + kKeys - 1) / kKeys * kKeys;
  const int64_t rows = (int64_t)batch * kt;
  const int64_t a = ((rows * kHeadDim * 2 + 255) / 256) * 256;
  const int64_t s = ((rows * 4 + 255) / 256) * 256;
  // ... and, last, the work-queue counters of the decode launch that takes a varlen batch's
  // one-token rows (see cai_mqa_prefill_varlen).
  return (size_t)(2 * a + 2 * s + ((piece_bytes() + 255) / 256) * 256 + kWorkspaceHeader);
}

// The piece region of a prefill workspace: a chunk call's prefill kernel writes the last
// wave's partial outputs there; a varlen call's prefill writes none, and its decode launch
// may keep its split partials there.
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
  p.compact = L.q_off ? 1 : 0;
  p.batch = L.batch;
  p.n_new = L.n_new;
  p.total_new = L.total_new;
  p.num_heads = L.num_heads;
  p.log2_heads = 31 - __builtin_clz((unsigned)L.num_heads);
  p.window = L.window;
  p.kt_rows = (int32_t)(((int64_t)L.max_pages * L.page_size + kKeys - 1) / kKeys * kKeys);
  p.qtiles = (int32_t)(((int64_t)L.n_new * L.num_heads + kQT * kRows - 1) / (kQT * kRows));
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

  const int64_t dq_blocks = (int64_t)L.batch * (p.kt_rows / kKeys);
  if (dq_blocks > 0 && L.q_off && L.batch <= kMaxCompactSeqs)
    dequant_compact_kernel<<<dim3((unsigned)std::min<int64_t>(dq_blocks, 4 * (int64_t)num_sms())), 256,
                             (L.batch + 1) * 4, stream>>>(p);
  else if (dq_blocks > 0)
    dequant_kernel<<<dim3((unsigned)(p.kt_rows / kKeys), (unsigned)L.batch), 256, 0, stream>>>(p);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;

  static bool attr_set[64] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 64 && !attr_set[dev]) {
    // The register split inside the kernel assumes the launch register count.
    cudaFuncAttributes fa;
    for (const void* fn : {(const void*)prefill_kernel<false>, (const void*)prefill_kernel<true>}) {
      e = cudaFuncGetAttributes(&fa, fn);
      if (e != cudaSuccess) return e;
      if (fa.numRegs != kRegsLaunch) return cudaErrorInvalidDeviceFunction;
      e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytesMax);
      if (e != cudaSuccess) return e;
    }
    attr_set[dev] = true;
  }
  // Work split (work_split) of a chunk call's q-tiles.  A varlen call's q-tiles are
  // counted on the device (whole, no pieces); the dense count here is the fallback when
  // they are too many to list.
  const int64_t qtiles_total = (int64_t)L.batch * p.qtiles;
  const int sms = num_sms();
  const int grid = (int)(qtiles_total < sms ? qtiles_total : sms);
  WorkSplit split = work_split(qtiles_total, grid);
  if (p.compact) split = WorkSplit{(int)qtiles_total, 1, (int)qtiles_total};
  p.pieces = split.pieces;
  p.full_items = split.full;
  p.num_items = split.num;
  const int smem = p.compact ? kSmemBytesMax : kSmemBytes;
  if (p.compact)
    prefill_kernel<true><<<grid, kThreads, smem, stream>>>(p);
  else
    prefill_kernel<false><<<grid, kThreads, smem, stream>>>(p);
  e = cudaGetLastError();
  if (e != cudaSuccess || split.pieces == 1) return e;
  const int64_t warps_c = (int64_t)(split.num - split.full) / split.pieces * kRows;  // one warp per row
  return launch_pdl(combine_pieces_kernel, dim3((unsigned)((warps_c + 7) / 8)), dim3(256), 0, stream, p);
}

}  // namespace cai
