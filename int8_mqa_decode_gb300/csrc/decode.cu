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
// How.  A persistent kernel, one CTA per SM, takes work items (layer,
// sequence, KV head, split; up to eight layers per launch, global layers'
// items first) from a global queue and walks each in 128-token tiles.  The scores
// are computed transposed, S^T = K Q^T (tokens x heads), so that one thread
// owns one token: its K and V scales and its mask are per-thread scalars and
// the K operand goes from registers to tensor memory without a shared-memory
// copy.  Warp roles, connected by mbarriers:
//  * scheduler (warp 2): claims items with an atomic counter, prefetches the
//    item's block-table lines into L2 and publishes the item, with the page
//    ids of its first tiles, into a small ring read by every role;
//  * producer (warp 0): per page, one 2-D tensor copy (TMA) of its K and V
//    code rows into a 128-byte-swizzled slot (so that reading one token row
//    per thread is free of bank conflicts) and one 1-D bulk copy of its two
//    scale rows, into a ring of 64-token stages.  Each lane issues one page.
//    Page ids are fetched a batch of tiles ahead, one id per lane.  Pages
//    wholly outside the split (the part of a local layer before its window)
//    are never read;
//  * converters (warps 4-11): read a tile's codes and scales into registers
//    and hand the stages back at once; then K codes -> fp16 (exact) into tensor
//    memory as the A operand of S^T (one token per lane), V codes -> fp16 into
//    tensor memory as the A operand V^T of PV (one channel per lane: a page
//    keeps its V codes channel-major, so a lane's 16-byte load holds 16 tokens
//    of its channel), the per-token scales and mask into a four-tile ring, and
//    at an item's first tile the item's query (bf16 -> fp16) as the K-major B
//    operand Q^T;
//  * MMA issuers: warp 1 issues S^T = K Q^T (tcgen05.mma kind::f16, M = 128
//    tokens, N = heads padded to 32 or 64, K = 128, A from tensor memory) into
//    a double-buffered S^T; warp 3 issues O^T += V^T P^T (M = 128 channels,
//    N = heads, K = 128 tokens, V^T from tensor memory, P^T from shared
//    memory) into one of two O^T accumulators (one per item in flight).  Each
//    launch of 8 K steps holds its issuing thread for most of its run time, so
//    the two streams are issued by different warps;
//  * softmax (warps 12-15, one thread per token of the tile): applies the K
//    scale and softmax scale, checks the logits against a per-head reference
//    maximum shared by the four warps (at an item's first tile, the logits of
//    its first attended token) that is raised only when a logit exceeds
//    it by 2^8 (one barrier-reduction per tile decides; O^T is rarely
//    rescaled), scales P by the token's V scale and stores it, fp16, as the
//    B operand P^T; at the end of an item it reduces the per-head sums and
//    writes the normalised output and its log-sum-exp (or the partial ones of
//    a split).
#include "common.cuh"
#include "ptx.cuh"
#include "tma.cuh"

namespace cai {
namespace {

constexpr int T = kDecodeTile;                 // 128 tokens per tile
constexpr int RT = 64;                         // tokens per raw stage
constexpr int kStageKV = RT * 2 * kHeadDim;    // K and V code rows of one stage (16 KB)
constexpr int kStageSc = RT * 8;               // their K and V scales (512 B)
constexpr int kRing = 6;                       // ring of published work items (readers lag the producer)
constexpr int kClaimAhead = 2;                 // items claimed but not yet started by the producer, at most
constexpr int kRingInts = 40;                  // ring entry: 8 item fields + 32 page ids
constexpr int kScaleSlots = 4;                 // scale/mask ring depth (tiles)

// Shared-memory layout for HN padded heads (32 or 64).
template <int HN>
struct Layout {
  static constexpr int NST = HN <= 32 ? 11 : 9;                  // raw stages
  static constexpr int kOffRawKV = 0;                            // [NST][16 KB], 1024-aligned (swizzle)
  static constexpr int kPTBytes = HN * T * 2;
  static constexpr int kOffPT = kOffRawKV + NST * kStageKV;      // P^T[2]
  static constexpr int kOffQT = kOffPT + 2 * kPTBytes;           // Q^T
  static constexpr int kOffRawSc = kOffQT + HN * kHeadDim * 2;   // [NST][512 B]
  static constexpr int kOffScal = kOffRawSc + NST * kStageSc;    // [4][T] float4s
  static constexpr int kOffXch = kOffScal + kScaleSlots * T * 16;  // softmax exchange, 13 x HN floats
  static constexpr int kOffBars = kOffXch + 13 * HN * 4;
  static_assert(kOffXch % 16 == 0 && kOffPT % 16 == 0, "bulk-copy sources");
  static constexpr int kNumBars = 2 * NST + 2 * 2 /*k_full, v_full*/ + 2 * 2 /*s_full, p_full*/ + 2 /*v_free*/ +
                                  2 * 2 /*o_full, o_empty*/ + 3 * kRing + 2 * kScaleSlots + 1 /*drain*/;
  static constexpr int kOffMisc = kOffBars + 8 * kNumBars;       // tmem slot, wait state (+8), page_ok[NST] (+24)
  static constexpr int kOffRing = kOffMisc + 80;
  static constexpr int kSmemBytes = kOffRing + kRing * kRingInts * 4 + 1024;
  static_assert(kSmemBytes <= 227 * 1024, "dynamic shared memory per CTA");
  static_assert(24 + 4 * NST <= 80, "misc words");
};

// Warp roles, aligned to warpgroups so each group can resize its register file:
//   warpgroup 0: producer (warp 0), S^T issuer (warp 1), scheduler (warp 2), PV issuer (warp 3)
//   warpgroups 1-2: converters (warps 4..11, two per TMEM lane quarter)
//   then softmax: one warp per lane quarter for up to 32 heads (warps 12..15), two
//   per lane quarter for 64 heads (warps 12..19, each taking half of the heads).
constexpr int kSchedWarp = 2;
constexpr int kConvWarp0 = 4;
constexpr int kConvWarps = 8;
constexpr int kSoftWarp0 = kConvWarp0 + kConvWarps;
template <int HN>
struct Roles {
  static constexpr int kSoftWarps = HN <= 32 ? 4 : 8;
  static constexpr int kThreads = 32 * (kSoftWarp0 + kSoftWarps);
  // Registers per thread, launched with kRegsLaunch and resized per warpgroup:
  //  32 heads: 16 warps (4 per SM sub-partition) at 128 = 65536; then 56 / 104 / 232:
  //            128 * (56 + 2 * 104 + 232) = 63488, per sub-partition 32 * 496 = 15872 <= 16384.
  //  64 heads: 20 warps (5 per sub-partition) at 96 = 61440; then 48 / 80 / 136:
  //            128 * (48 + 2 * 80 + 2 * 136) = 61440, per sub-partition 32 * 480 = 15360 <= 16384
  //            (the softmax holds 32 heads per thread; below 136 registers it spills).
  static constexpr int kRegsLaunch = HN <= 32 ? 128 : 96;  // checked on the host before the first launch
  static constexpr int kRegsCtl = HN <= 32 ? 56 : 48;
  static constexpr int kRegsConv = HN <= 32 ? 104 : 80;
  static constexpr int kRegsSoft = HN <= 32 ? 232 : 136;
  static_assert(128 * kRegsCtl + 32 * kConvWarps * kRegsConv + 32 * kSoftWarps * kRegsSoft <= kRegsLaunch * kThreads,
                "register split");
  static_assert(32 * (kRegsCtl + 2 * kRegsConv + (kSoftWarps / 4) * kRegsSoft) <= 16384, "sub-partition registers");
  static_assert((kThreads / 32 + 3) / 4 * 32 * kRegsLaunch <= 16384, "launch registers per sub-partition");
  static constexpr int kItemReaders = 3 + kConvWarps + kSoftWarps;  // producer, 2 MMA, converters, softmax
};
constexpr int kNoPage = -2147483647 - 1;      // a page the tile does not need
constexpr uint32_t kTmemCols = 512;
constexpr float kRescaleThreshold = 8.0f;     // log2 units: weights stay <= 2^8 between rescales
constexpr float kFirstRefMargin = 6.0f;       // log2 units above an item's first token (see the softmax)
constexpr uint32_t kSoftBar = 1;              // named barrier of the softmax warpgroup

__device__ __forceinline__ void set_err(int32_t* err, int bits) {
  if (err) atomicOr(err, bits);
}

// Lane `lane` of a warp ends with the reduction over the warp of v[lane % N]
// (a reduce-scatter: N - 1 shuffles, plus one when N = 16).  Destroys v.
template <bool kMax, int N>
__device__ __forceinline__ float reduce_scatter(float (&v)[N], int lane) {
#pragma unroll
  for (int o = N / 2; o >= 1; o >>= 1) {
    const bool up = (lane & o) != 0;
#pragma unroll
    for (int i = 0; i < o; ++i) {
      const float send = up ? v[i] : v[i + o];
      const float keep = up ? v[i + o] : v[i];
      const float recv = __shfl_xor_sync(0xffffffffu, send, o);
      v[i] = kMax ? fmaxf(keep, recv) : keep + recv;
    }
  }
  float r = v[0];
#pragma unroll
  for (int o = 16; o >= N; o >>= 1) {
    const float x = __shfl_xor_sync(0xffffffffu, r, o);
    r = kMax ? fmaxf(r, x) : r + x;
  }
  return r;
}

// Lane i (< N) ends with the maximum over the warp of v[i]: one warp-wide float
// reduction (redux.sync, sm_100 family) per element.
template <int N>
__device__ __forceinline__ float warp_max_scatter(const float (&v)[N], int lane) {
  float r = -INFINITY;
#pragma unroll
  for (int i = 0; i < N; ++i) {
    float m;
    asm volatile("redux.sync.max.f32 %0, %1, 0xffffffff;" : "=f"(m) : "f"(v[i]));
    r = lane == i ? m : r;
  }
  return r;
}

// A work item: one split of one sequence of one layer (job).  kind 0 = tiles to
// process, 1 = nothing to attend (split 0 writes out = 0, lse = -inf).
struct Item {
  int job, b, kvh, split, start, end, tile0, ntiles;
  bool direct;  // single split: write the final output
  int kind;
  bool invalid;
};

// Ring entry: [0] b, [1] split, [2] start, [3] end, [4] tile0, [5] ntiles,
// [6] flags (bit 0 direct, bit 1 invalid, bit 2 kind 1, bit 3 end of work, bits 4.. job), [7] KV head,
// [8 .. 40) page ids of the item's first tiles (one id batch, see batch_page).
__device__ __forceinline__ Item ring_item(const volatile int32_t* e, bool& done) {
  Item it;
  it.b = e[0];
  it.split = e[1];
  it.start = e[2];
  it.end = e[3];
  it.tile0 = e[4];
  it.ntiles = e[5];
  const int f = e[6];
  it.kvh = e[7];
  it.direct = f & 1;
  it.invalid = (f >> 1) & 1;
  it.kind = (f >> 2) & 1;
  done = (f >> 3) & 1;
  it.job = f >> 4;
  return it;
}

// Page id of page slot `ps` of tile `t` of an item, or kNoPage if the tile does not need it.
template <int P>
__device__ __forceinline__ int32_t tile_page(const DecodeParams& p, const Item& it, int t, int ps) {
  const int t0 = (it.tile0 + t) * T + ps * P;
  if (t0 + P <= it.start || t0 >= it.end) return (int32_t)kNoPage;
  const DecodeJob& jb = p.job[it.job];
  return jb.table[(int64_t)it.b * jb.max_pages + t0 / P];
}

// Id batch `batch` of an item: lane l holds page slot l % (T/P) of tile
// batch * (32 / (T/P)) + l / (T/P).
template <int P>
__device__ __forceinline__ int32_t batch_page(const DecodeParams& p, const Item& it, int batch, int lane) {
  constexpr int PPT = T / P, TPB = 32 / PPT;
  const int t = batch * TPB + lane / PPT;
  return t < it.ntiles ? tile_page<P>(p, it, t, lane % PPT) : (int32_t)kNoPage;
}

// Work item idx: the job whose range holds it, then, within the job,
// (b * num_kv_heads + kv head) * max_splits + split.  kind 2 = an empty split, never published.
template <int P>
__device__ __forceinline__ Item make_item(const DecodeParams& p, int idx) {
  Item it;
  int j = 0;
  while (j + 1 < p.num_jobs && idx >= p.job[j + 1].item0) ++j;
  const DecodeJob& jb = p.job[j];
  it.job = j;
  idx -= jb.item0;
  const int per_b = p.num_kv_heads * jb.plan.max_splits;
  it.b = idx / per_b;
  const int r = idx - it.b * per_b;
  it.kvh = r / jb.plan.max_splits;
  it.split = r - it.kvh * jb.plan.max_splits;
  int32_t L = p.ctx_len[it.b];
  if (jb.q_off) {
    const int32_t a = jb.q_off[it.b], e = jb.q_off[it.b + 1];
    if (!(a >= 0 && e == a + 1 && e <= jb.total_rows)) {  // not a one-token row: the prefill kernel's
      it.kind = 2;
      it.invalid = false;
      it.direct = false;
      it.ntiles = 0;
      it.start = it.end = it.tile0 = 0;
      return it;
    }
    L = L + 1;  // ctx_len holds the prefix length; the new token is attended too
  }
  const SeqSplits sp = seq_splits(L, jb.window, jb.max_pages * P, jb.plan.chunk);
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
  it.start = sp.lo + it.split * jb.plan.chunk;
  it.end = min(sp.hi, it.start + jb.plan.chunk);
  it.tile0 = it.start / T;
  it.ntiles = (it.end - 1) / T - it.tile0 + 1;
  return it;
}

struct DecodeArgs {
  DecodeParams p;
  CUtensorMap kv_map[kMaxKvHeads];  // each pool slot as rows of 128 bytes; box = the 2P code rows of a page
};

template <int P, int HN>
__global__ void __launch_bounds__(Roles<HN>::kThreads, 1) decode_kernel(const __grid_constant__ DecodeArgs args) {
  using L = Layout<HN>;
  using R = Roles<HN>;
  constexpr int kSoftWarps = R::kSoftWarps;
  constexpr int NST = L::NST;
  constexpr int PPT = T / P;                   // pages per tile
  constexpr int TPB = 32 / PPT;                // tiles per page-id batch
  constexpr int SPS = RT / P;                  // pages per stage
  constexpr int kRowsPerPage = page_bytes(P) / 128;
  constexpr uint32_t kColKA = 0;               // K operand [2]: 64 columns each (fp16 pairs)
  constexpr uint32_t kColV = 128;              // V^T operand [2]: 64 columns each (fp16 token pairs)
  constexpr uint32_t kColS = 256;              // S^T [2]: HN columns each
  constexpr uint32_t kColO = 256 + 2 * HN;     // O^T [2]: HN columns each
  static_assert(kColO + 2 * HN <= kTmemCols, "tensor memory columns");
  static_assert(page_bytes(P) % 128 == 0 && P % 16 == 0, "page rows");
  const DecodeParams& p = args.p;

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* raw_kv = smem + L::kOffRawKV;
  uint8_t* raw_sc = smem + L::kOffRawSc;
  uint8_t* pt = smem + L::kOffPT;
  uint8_t* qt = smem + L::kOffQT;
  float4* scal = reinterpret_cast<float4*>(smem + L::kOffScal);  // [kScaleSlots][T] (k scale, valid, v scale, 0)
  float* xch = reinterpret_cast<float*>(smem + L::kOffXch);
  float* wmax = xch;              // [4][HN] per-warp maxima
  float* lpart = xch + 4 * HN;    // [4][HN] per-warp sums
  float* mref = xch + 8 * HN;     // [HN] reference maxima (-inf: none yet)
  float* muse = mref + HN;        // [HN] the reference as subtracted (0 when none)
  float* aref = muse + HN;        // [HN] rescale factors of the last raise
  float* dref = aref + HN;        // [HN] shift of the subtracted reference at the last raise
  float* linv = dref + HN;        // [HN] 1 / row sums
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::kOffBars);
  uint64_t* raw_full = bars;                 // [NST] producer -> converters (tx bytes)
  uint64_t* raw_empty = bars + NST;          // [NST] converters -> producer
  uint64_t* k_full = bars + 2 * NST;         // [2] converters -> MMA (K operand, Q^T)
  uint64_t* v_full = k_full + 2;             // [2] converters -> MMA (V^T operand)
  uint64_t* s_full = v_full + 2;             // [2] MMA commit after S^T
  uint64_t* p_full = s_full + 2;             // [2] softmax -> MMA (P^T)
  uint64_t* v_free = p_full + 2;             // [2] MMA commit after PV (V^T and P^T free)
  uint64_t* o_full = v_free + 2;             // [2] MMA commit after an item's last PV
  uint64_t* o_empty = o_full + 2;            // [2] softmax -> MMA after reading O^T
  uint64_t* item_full = o_empty + 2;         // [kRing] scheduler -> readers
  uint64_t* item_empty = item_full + kRing;  // [kRing] readers -> scheduler
  uint64_t* scale_full = item_empty + kRing;        // [kScaleSlots] converters -> softmax
  uint64_t* scale_free = scale_full + kScaleSlots;  // [kScaleSlots] softmax -> converters
  uint64_t* item_taken = scale_free + kScaleSlots;  // [kRing] producer -> scheduler (item started)
  uint64_t* mma_drain = item_taken + kRing;         // MMA issuers' last commits, at exit
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::kOffMisc);
  volatile WaitState* const wctl = reinterpret_cast<volatile WaitState*>(smem + L::kOffMisc + 8);
  volatile int32_t* abort_flag = &wctl->abort;
  uint32_t* page_ok = reinterpret_cast<uint32_t*>(smem + L::kOffMisc + 24);        // [NST]
  volatile int32_t* ring = reinterpret_cast<volatile int32_t*>(smem + L::kOffRing);  // [kRing][kRingInts]

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int Hq = p.num_heads;                   // query heads per sequence (row stride of q and out)
  const int G = Hq / p.num_kv_heads;            // query heads per KV head (the rows of one item)
  const int num_items = p.num_items;

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
      mbar_init(&o_full[c], 1);
      mbar_init(&o_empty[c], kSoftWarps);
    }
    for (int r = 0; r < kRing; ++r) {
      mbar_init(&item_full[r], 1);
      mbar_init(&item_empty[r], R::kItemReaders);
      mbar_init(&item_taken[r], 1);
    }
    mbar_init(mma_drain, 2);
    for (int r = 0; r < kScaleSlots; ++r) {
      mbar_init(&scale_full[r], kConvWarps);
      mbar_init(&scale_free[r], kSoftWarps);
    }
    *abort_flag = 0;
    wctl->limit_ns = p.wait_ns;
    fence_barrier_init();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  // Everything above touched only this CTA's own resources; from here on the kernel
  // reads and writes memory that the previous kernels in the stream may still use.
  if (!p.overlap_prev) grid_dependency_wait();
  grid_launch_dependents();

  // Item k of this CTA as published by the scheduler warp; every reader warp
  // waits for it, copies it and releases the slot.  Waits answer per thread (no
  // collective step right after a wait on the hot path, where one costs about 15% of
  // the decode), so the reader's lanes agree here, once per item: the item is used
  // only if every lane saw it published and none has given up earlier (`stop`);
  // otherwise `done` ends the reader.  The softmax warps agree through their own
  // barrier-reduction instead (group_vote = false: `done` is then per lane).
  auto next_item = [&](int k, bool& done, bool stop, bool group_vote, int32_t* first_ids = nullptr) -> Item {
    const int slot = k % kRing;
    const bool seen = mbar_wait_abortable(&item_full[slot], (k / kRing) & 1, wctl);
    Item it = ring_item(ring + slot * kRingInts, done);
    if (first_ids) *first_ids = (int32_t)ring[slot * kRingInts + 8 + lane];
    __syncwarp();
    if (lane == 0 && seen) {  // a slot is released only by a reader that saw it published
      mbar_arrive(&item_empty[slot]);
      if (warp == 0) mbar_arrive(&item_taken[slot]);  // the producer starts item k
    }
    if (group_vote ? !__all_sync(0xffffffffu, seen && !stop) : !(seen && !stop)) done = true;
    return it;
  };
  if (warp < kConvWarp0) {
    setmaxnreg_dec<R::kRegsCtl>();
    if (warp == kSchedWarp) {
      // ---------------------------------------------------------- scheduler
      // An item is claimed from the global queue only once the producer has started the
      // item kClaimAhead before it: a CTA holds few claimed items, so the queue, not
      // early claims, decides which SM runs what (claiming up to the ring's depth let
      // a few SMs hoard long items and finish far behind the others).
      // Lane 0 decides for the warp (the claim goes through a shuffle); a lane writes
      // its part of a ring slot only after seeing every reader release the slot.
      int k = 0;
      bool stop = false;  // lane 0: one of its waits gave up
      while (true) {
        const bool taken = k < kClaimAhead || mbar_wait_abortable(&item_taken[(k - kClaimAhead) % kRing],
                                                                  ((k - kClaimAhead) / kRing) & 1, wctl);
        int idx = -1;
        if (lane == 0 && taken && !stop) idx = (int)atomicAdd(&p.queue[0], 1u);
        idx = __shfl_sync(0xffffffffu, idx, 0);
        if (idx < 0) break;
        const bool done = idx >= num_items;
        Item it = {};
        int32_t id = (int32_t)kNoPage;
        if (!done) {
          it = make_item<P>(p, idx);
          if (it.kind == 2) continue;  // an empty split: nobody needs to hear of it
          if (it.kind == 0) {
            id = batch_page<P>(p, it, 0, lane);
            // Warm L2 with the item's block-table entries (32 ids per 128-byte line, one line per lane).
            const int first = it.start / P, last = (it.end - 1) / P;
            const int32_t* row = p.job[it.job].table + (int64_t)it.b * p.job[it.job].max_pages;
            for (int pg = (first & ~31) + lane * 32; pg <= last; pg += 32 * 32) prefetch_l2(row + pg);
          }
        }
        const int slot = k % kRing;
        const bool free = k < kRing || mbar_wait_abortable(&item_empty[slot], ((k / kRing) - 1) & 1, wctl);
        volatile int32_t* e = ring + slot * kRingInts;
        if (free) e[8 + lane] = id;
        if (lane == 0 && free) {
          if (!done) {
            e[0] = it.b;
            e[1] = it.split;
            e[2] = it.start;
            e[3] = it.end;
            e[4] = it.tile0;
            e[5] = it.ntiles;
            e[6] = (it.direct ? 1 : 0) | (it.invalid ? 2 : 0) | (it.kind == 1 ? 4 : 0) | (it.job << 4);
            e[7] = it.kvh;
          } else {
            e[6] = 8;
          }
        }
        __syncwarp();
        if (lane == 0) {
          if (free) {
            __threadfence_block();
            mbar_arrive(&item_full[slot]);
          } else {
            stop = true;
          }
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
      // ---------------------------------------------------------- producer
      // `ids` holds the current batch of page ids (one per lane), `ids_next` the
      // following batch, loaded a whole batch of tiles before it is needed.
      const uint64_t policy = policy_evict_first();
      int r = 0, k = 0;
      while (true) {
        bool done = false;
        int32_t ids = kNoPage;
        const Item it = next_item(k++, done, *abort_flag != 0, true, &ids);
        if (done) break;
        if (it.kind != 0) continue;
        bool ok = true;
        const int slot = p.job[it.job].slot0 + it.kvh;
        const CUtensorMap* kv_map = &args.kv_map[slot];
        const uint8_t* pages = p.pages[slot];
        const int slot_pages = p.slot_pages[slot];
        int32_t ids_next = it.ntiles > TPB ? batch_page<P>(p, it, 1, lane) : (int32_t)kNoPage;
        for (int t = 0; t < it.ntiles && ok; ++t) {
          if (t > 0 && t % TPB == 0) {
            ids = ids_next;
            ids_next = t + TPB < it.ntiles ? batch_page<P>(p, it, t / TPB + 1, lane) : (int32_t)kNoPage;
          }
          for (int hf = 0; hf < 2; ++hf, ++r) {
            const int s = r % NST;
            // The warp reaches the wait converged (nothing in this loop branches on the
            // lane: the copies below are predicated), so its one wait instruction stream
            // gives every lane the same answer and the lanes leave together.  (A
            // collective step right after this wait, to agree explicitly, costs about
            // 5% of the decode: the stage turnaround is on the critical path.)
            if (r >= NST && !mbar_wait_abortable(&raw_empty[s], ((r / NST) - 1) & 1, wctl)) {
              ok = false;
              break;
            }
            const int32_t pid = __shfl_sync(0xffffffffu, ids, (t % TPB) * PPT + hf * SPS + lane % SPS);
            const bool live = lane < SPS && pid != kNoPage;
            const bool in_range = pid >= 0 && pid < slot_pages;
            if (live && !in_range) set_err(p.err, CAI_DEVERR_PAGE);
            const uint32_t okm = __ballot_sync(0xffffffffu, live && in_range);
            if (lane == 0) {
              page_ok[s] = okm;
              // (Fault injection: the dropped stage expects 16 bytes that never come.)
              mbar_arrive_expect_tx(&raw_full[s], (uint32_t)__popc(okm) * page_bytes(P) + (r == p.drop_stage ? 16u : 0u));
            }
            __syncwarp();
            const bool mine = (okm >> lane) & 1u;
            const int32_t pg = mine ? pid : 0;
            tma_load_2d_hint_if(mine, raw_kv + s * kStageKV + lane * (2 * P * kHeadDim), kv_map, 0, pg * kRowsPerPage,
                                &raw_full[s], policy);
            bulk_g2s_hint_if(mine, raw_sc + s * kStageSc + lane * (8 * P), pages + (int64_t)pg * page_bytes(P) + 2 * P * kHeadDim,
                             8 * P, &raw_full[s], policy);
          }
        }
        if (!ok) break;
      }
      // Every stage this producer armed has landed before the CTA goes away, whatever
      // happened to the other roles (copies into a CTA's shared memory must not outlive it).
      for (int i = r > NST ? r - NST : 0; i < r; ++i)
        if (i != p.drop_stage) mbar_wait_drain(&raw_full[i % NST], (i / NST) & 1);
    } else {
      // ---------------------------------------------------------- MMA issuers
      // Warp 1 issues S^T = K Q^T, warp 3 issues O^T += V^T P^T: each waits only for
      // its own operands, so one warp's barrier waits overlap the other's launches,
      // and an item's last PV goes out as soon as its P^T is ready.
      constexpr uint32_t idesc_s = idesc_f16_f32(T, HN, 0, 0);
      constexpr uint32_t idesc_o = idesc_f16_f32(kHeadDim, HN, 0, 1);  // A = V^T from tensor memory
      // Descriptor bases; a K step of 16 adds 256 bytes, i.e. 16 to the address field
      // (shared addresses stay below 2^18, so the 14-bit field never carries).
      const uint64_t dq = smem_desc(smem_addr(qt), 128, 2048);
      const uint64_t dp = smem_desc(smem_addr(pt), 128, T * 16);
      const bool s_issuer = warp == 1;
      // Every lane runs the loop and waits for itself; lane 0 issues only what its own
      // waits allow.  The lanes agree at the end of each tile (one vote, which also
      // keeps them together while lane 0 issues).
      int g = 0, item_n = 0, k = 0;
      bool ok = true;
      while (true) {
        bool done = false;
        const Item it = next_item(k++, done, !ok, true);
        if (done) break;
        if (it.kind != 0) continue;
        const int ob = item_n & 1;
        for (int t = 0; t < it.ntiles; ++t, ++g) {
          const int c = g & 1;
          if (s_issuer) {
            // S^T[c] is free once the softmax of tile g-2 has read it (it then wrote P^T).
            ok = mbar_wait_abortable(&k_full[c], (g >> 1) & 1, wctl) &&
                 (g < 2 || mbar_wait_abortable(&p_full[c], ((g >> 1) - 1) & 1, wctl));
            tc_fence_after();
            if (lane == 0 && ok) {
#pragma unroll
              for (int ks = 0; ks < kHeadDim / 16; ++ks)
                mma_f16_ts(tmem + kColS + c * HN, tmem + kColKA + c * 64 + ks * 8, dq + (uint64_t)(ks * 16), idesc_s,
                           ks > 0 ? 1u : 0u);
              mma_commit(&s_full[c]);
            }
          } else {
            // PV of tile g into O^T[item & 1]; the item's first PV starts the
            // accumulator once the epilogue of item - 2 has read it.
            ok = mbar_wait_abortable(&p_full[c], (g >> 1) & 1, wctl) &&
                 mbar_wait_abortable(&v_full[c], (g >> 1) & 1, wctl) &&
                 (t > 0 || item_n < 2 || mbar_wait_abortable(&o_empty[ob], ((item_n >> 1) - 1) & 1, wctl));
            tc_fence_after();
            if (lane == 0 && ok) {
#pragma unroll
              for (int ks = 0; ks < T / 16; ++ks)
                mma_f16_ts(tmem + kColO + ob * HN, tmem + kColV + c * 64 + ks * 8,
                           dp + (uint64_t)(c * (L::kPTBytes >> 4) + ks * 16), idesc_o, (t > 0 || ks > 0) ? 1u : 0u);
              mma_commit(&v_free[c]);
              if (t == it.ntiles - 1) mma_commit(&o_full[ob]);
            }
          }
          ok = __all_sync(0xffffffffu, ok);
          if (!ok) break;
        }
        ++item_n;
      }
      // This issuer's MMAs have completed before tensor memory is freed.
      if (lane == 0) {
        mma_commit(mma_drain);
        mbar_wait_drain(mma_drain, 0);
      }
      __syncwarp();
    }
  } else if (warp < kSoftWarp0) {
    setmaxnreg_dec<R::kRegsConv>();
    // ------------------------------------------------------------ converters
    const int ctid = tid - kConvWarp0 * 32;           // 0 .. 255
    const int quarter = warp & 3;                     // TMEM lanes this warp may touch
    const int hh = (warp - kConvWarp0) >> 2;          // which 64 channels of its token's K
    const int tk = quarter * 32 + lane;               // this thread's token (K operand row)
    const uint32_t t_lane = (uint32_t)(quarter * 32) << 16;
    constexpr int kQUnits = HN * 16 / 256;            // 16-byte units of Q^T per thread
    // A converter warp's control flow does not depend on its waits: a lane whose wait
    // gave up carries on with the tile (its operands are then garbage) and releases
    // nothing it did not see filled; the lanes agree on stopping at the next item.
    int g = 0, k = 0;
    bool ok = true;
    while (true) {
      bool done = false;
      const Item it = next_item(k++, done, !ok, true);
      if (done) break;
      if (it.kind != 0) continue;
      // The item's query as Q^T (bf16 -> fp16), once the S^T of the previous
      // item's last tile (g-1), which reads the old one, is done.
      // Unit u: head n (8 consecutive lanes take 8 consecutive heads), channels 8*k8 .. 8*k8 + 7.
      {
        uint4 qv[kQUnits];
#pragma unroll
        for (int i = 0; i < kQUnits; ++i) {
          const int u = i * 256 + ctid;
          const int n = (u & 7) | ((u >> 7) << 3), k8 = (u >> 3) & 15;
          qv[i] = n < G ? __ldg(reinterpret_cast<const uint4*>(p.job[it.job].q + (job_row(p.job[it.job], it.b) * Hq + it.kvh * G + n) * kHeadDim +
                                                                k8 * 8))
                        : make_uint4(0u, 0u, 0u, 0u);
        }
        if (g >= 1) ok = mbar_wait_abortable(&s_full[(g - 1) & 1], ((g - 1) >> 1) & 1, wctl) && ok;
#pragma unroll
        for (int i = 0; i < kQUnits; ++i) {
          const int u = i * 256 + ctid;
          const int n = (u & 7) | ((u >> 7) << 3), k8 = (u >> 3) & 15;
          const uint32_t xs[4] = {qv[i].x, qv[i].y, qv[i].z, qv[i].w};
          uint32_t o[4];
#pragma unroll
          for (int e = 0; e < 4; ++e)
            o[e] = pack_f16x2(__uint_as_float(xs[e] << 16), __uint_as_float(xs[e] & 0xFFFF0000u));
          *reinterpret_cast<uint4*>(qt + (n >> 3) * 2048 + k8 * 128 + (n & 7) * 16) = make_uint4(o[0], o[1], o[2], o[3]);
        }
        fence_proxy_async_smem();
      }
      for (int t = 0; t < it.ntiles; ++t, ++g) {
        const int c = g & 1;
        const int s0 = (2 * g) % NST, s1 = (2 * g + 1) % NST;
        // Only a lane that saw both stages land may release them (lane 0 does).
        const bool landed = mbar_wait_abortable(&raw_full[s0], ((2 * g) / NST) & 1, wctl) &&
                            mbar_wait_abortable(&raw_full[s1], ((2 * g + 1) / NST) & 1, wctl);
        ok = ok && landed;
        // Codes to registers.  Row r of a page slot holds its 16-byte chunk j at
        // chunk position j ^ (r % 8) (128-byte swizzle; slots are 1024-aligned,
        // and a page occupies 2P rows of its stage, a multiple of 8).
        //  K: this thread's token tk, channels hh*64 .. hh*64+63 (K rows are token-major).
        //  V: this thread's channel tk, the 64 tokens of tile half hh (stage s0 or s1):
        //     V rows are channel-major, so 16 consecutive tokens of one channel are one
        //     16-byte chunk: channel c's codes start at byte c*P of the page's V block
        //     (block rows P .. 2P-1 of the page).
        uint4 wk[4], wv[4];
        {
          const int tr = tk & (RT - 1);
          const uint8_t* row = raw_kv + (tk < RT ? s0 : s1) * kStageKV + (tr / P) * (2 * P * kHeadDim) +
                               (tr % P) * kHeadDim;
#pragma unroll
          for (int i = 0; i < 4; ++i) wk[i] = *reinterpret_cast<const uint4*>(row + (((hh * 4 + i) ^ (tk & 7)) << 4));
        }
        {
          const uint8_t* st = raw_kv + (hh ? s1 : s0) * kStageKV;
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            const int j = (u * 16) / P, o = (u * 16) % P;       // page of the stage, first token in it
            const int off = tk * P + o;                          // byte within the page's V block
            const int r = P + off / 128, ch = (off % 128) / 16;  // row of the page, chunk of the row
            wv[u] = *reinterpret_cast<const uint4*>(st + j * (2 * P * kHeadDim) + r * 128 + ((ch ^ (r & 7)) << 4));
          }
        }
        // Scales and mask of tile g into ring slot g % 4 (free once the softmax of tile g-4 is done).
        const int ss = g & (kScaleSlots - 1);
        if (g >= kScaleSlots) ok = mbar_wait_abortable(&scale_free[ss], ((g / kScaleSlots) - 1) & 1, wctl) && ok;
        if (ctid < T) {
          const int tt = ctid;
          const int s = tt < RT ? s0 : s1;
          const int tr = tt & (RT - 1);
          const int abs_t = (it.tile0 + t) * T + tt;
          const bool valid = abs_t >= it.start && abs_t < it.end && ((page_ok[s] >> (tr / P)) & 1u);
          const float* sc = reinterpret_cast<const float*>(raw_sc + s * kStageSc + (tr / P) * (8 * P));
          scal[ss * T + tt] = valid ? make_float4(sc[tr % P] * p.scale_log2, 1.0f, sc[P + tr % P], 0.0f)
                                    : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
        }
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(&scale_full[ss]);
          if (landed) {
            mbar_arrive(&raw_empty[s0]);
            mbar_arrive(&raw_empty[s1]);
          }
        }
        // K -> tensor memory: K[c] is free once S^T of tile g-2 is done.
        if (g >= 2) ok = mbar_wait_abortable(&s_full[c], ((g >> 1) - 1) & 1, wctl) && ok;
        tc_fence_after();
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          uint32_t kw[16];
#pragma unroll
          for (int i = 0; i < 2; ++i) {
            const uint4 w = wk[half * 2 + i];
            const uint32_t xs[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) i8x4_to_f16x4(xs[e], kw[(i * 4 + e) * 2], kw[(i * 4 + e) * 2 + 1]);
          }
          tmem_st_32x32b_x16(tmem + t_lane + kColKA + c * 64 + hh * 32 + half * 16, kw);
        }
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&k_full[c]);
        // V -> V^T[c] in tensor memory (lane = channel, column k = tokens 2k, 2k+1 of
        // the tile; this warp writes the 32 columns of its tile half), free once PV of
        // tile g-2 is done.
        if (g >= 2) ok = mbar_wait_abortable(&v_free[c], ((g >> 1) - 1) & 1, wctl) && ok;
        tc_fence_after();
        {
          uint32_t vw[32];
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            const uint32_t xs[4] = {wv[u].x, wv[u].y, wv[u].z, wv[u].w};
#pragma unroll
            for (int e = 0; e < 4; ++e) i8x4_to_f16x4(xs[e], vw[u * 8 + e * 2], vw[u * 8 + e * 2 + 1]);
          }
          tmem_st_32x32b_x32(tmem + t_lane + kColV + c * 64 + hh * 32, vw);
        }
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&v_full[c]);
      }
    }
  } else {
    setmaxnreg_inc<R::kRegsSoft>();
    // ------------------------------------------------------------ softmax + epilogue
    // Thread = token tok of each tile (TMEM lane of S^T) and channel tok of O^T;
    // warp half hp takes heads [hp * HH, hp * HH + HH).
    constexpr int HH = HN / (kSoftWarps / 4);
    constexpr uint32_t kSoftThreads = 32 * kSoftWarps;
    const int sw = warp - kSoftWarp0;
    const int quarter = warp & 3;
    const int hp = sw >> 2;
    const int h0 = hp * HH;
    const int tok = quarter * 32 + lane;
    const uint32_t t_lane = (uint32_t)(quarter * 32) << 16;
    // The softmax warps meet at named barriers, so they stop together.  A thread
    // whose wait gave up carries on with the same steps (on garbage) and brings
    // ok = false to the group's next barrier-reduction (the item's start, a raise,
    // the item's end), which gives every thread the same answer.
    int g = 0, item_n = 0, k = 0;
    bool ok = true;
    while (true) {
      bool done = false;
      const Item it = next_item(k++, done, false, false);
      if (bar_red_or(kSoftBar, kSoftThreads, done)) break;
      // The previous item's bulk copies must have read the P^T buffers and the
      // exchange before this item writes them; every softmax thread passes the
      // first tile's barrier-reduction after this.
      if (sw == 0 && lane == 0) bulk_wait_read_all();
      if (it.kind == 1) {
        // Nothing to attend (L = 0) or an invalid length: out = 0, lse = -inf.
        if (it.invalid && sw == 0 && lane == 0) set_err(p.err, CAI_DEVERR_LENGTH);
        const DecodeJob& jb = p.job[it.job];
        const int64_t hb = job_row(jb, it.b) * Hq + it.kvh * G;  // first output head of the item
        for (int h = h0; h < h0 + HH && h < G; ++h) jb.out[(hb + h) * kHeadDim + tok] = 0.0f;
        if (jb.lse_out && quarter == 0 && lane < HH && h0 + lane < G) jb.lse_out[hb + h0 + lane] = -INFINITY;
        continue;
      }
      float l[HH];
#pragma unroll
      for (int h = 0; h < HH; ++h) l[h] = 0.0f;
      for (int t = 0; t < it.ntiles; ++t, ++g) {
        const int c = g & 1;
        const int ss = g & (kScaleSlots - 1);
        ok = ok && mbar_wait_abortable(&s_full[c], (g >> 1) & 1, wctl) &&
             mbar_wait_abortable(&scale_full[ss], (g / kScaleSlots) & 1, wctl);
        tc_fence_after();
        float sv[HH];
        {
          uint32_t r[HH];
          if constexpr (HH == 32) tmem_ld_32x32b_x32(tmem + t_lane + kColS + c * HN + h0, r);
          else tmem_ld_32x32b_x16(tmem + t_lane + kColS + c * HN + h0, r);
          tmem_wait_ld();
#pragma unroll
          for (int i = 0; i < HH; ++i) sv[i] = __uint_as_float(r[i]);
        }
        const float4 sc = scal[ss * T + tok];
        const float ks = sc.x;
        const bool valid = sc.y != 0.0f;
        const float vs = sc.z;
        if (t == 0) {
          // A new item's references: the logits of its first attended token plus a margin,
          // shared by the thread that holds it (-inf when that token is masked: the raise
          // below then sets them); a later logit above them by more than 2^8 raises them as
          // usual.  The margin makes such raises, which wait for the previous PV to rescale
          // O^T, rare: a logit 2^6 above the token's still leaves the weights <= 2^8.
          if (tok == it.start - it.tile0 * T) {
#pragma unroll
            for (int h = 0; h < HH; ++h) {
              const float z = sv[h] * ks + kFirstRefMargin;
              mref[h0 + h] = valid ? z : -INFINITY;
              muse[h0 + h] = valid ? z : 0.0f;
            }
          }
          named_barrier_sync(kSoftBar, kSoftThreads);
        }
        // e_h = logit (log2 units) minus the head's reference.
        float mx = -INFINITY;
        if (valid) {
          // Packed fp32 pairs: two FFMAs per instruction.
          const uint64_t ks2 = f2(ks, ks);
#pragma unroll
          for (int h = 0; h < HH; h += 4) {
            const float4 mu = *reinterpret_cast<const float4*>(muse + h0 + h);
            f2_split(f2_fma(f2(sv[h], sv[h + 1]), ks2, f2(-mu.x, -mu.y)), sv[h], sv[h + 1]);
            f2_split(f2_fma(f2(sv[h + 2], sv[h + 3]), ks2, f2(-mu.z, -mu.w)), sv[h + 2], sv[h + 3]);
            mx = fmax3(mx, fmax3(sv[h], sv[h + 1], sv[h + 2]), sv[h + 3]);
          }
        }
        // (A thread that gave up asks for a raise, and then all stop at its second reduction.)
        const bool raise = !ok || (valid && (mx > kRescaleThreshold || mref[h0] == -INFINITY));  // or no reference yet
        if (bar_red_or(kSoftBar, kSoftThreads, raise)) {
          if (bar_red_or(kSoftBar, kSoftThreads, !ok)) {
            ok = false;
            break;
          }
          // Some head's reference must rise (or none is set yet): per-head maxima of the
          // tile over the four lane quarters, new references.
          {
            float v[HH];
#pragma unroll
            for (int i = 0; i < HH; ++i) v[i] = valid ? sv[i] + muse[h0 + i] : -INFINITY;
            const float wm = warp_max_scatter<HH>(v, lane);
            if (lane < HH) wmax[quarter * HN + h0 + lane] = wm;
          }
          named_barrier_sync(kSoftBar, kSoftThreads);
          if (quarter == 0 && lane < HH) {
            const int h = h0 + lane;
            const float M = fmaxf(fmaxf(wmax[h], wmax[HN + h]), fmaxf(wmax[2 * HN + h], wmax[3 * HN + h]));
            const float m_old = mref[h];
            const float m_new = M > m_old + kRescaleThreshold ? M : m_old;
            const float mu_old = muse[h];
            const float mu_new = m_new == -INFINITY ? 0.0f : m_new;
            aref[h] = m_old == -INFINITY ? 0.0f : ex2_approx(m_old - m_new);
            dref[h] = mu_old - mu_new;
            mref[h] = m_new;
            muse[h] = mu_new;
          }
          named_barrier_sync(kSoftBar, kSoftThreads);
#pragma unroll
          for (int h = 0; h < HH; ++h) {
            l[h] *= aref[h0 + h];
            sv[h] += dref[h0 + h];
          }
          if (t > 0) {
            // O^T holds earlier tiles of this item: wait for the previous PV, then rescale this thread's entries.
            ok = mbar_wait_abortable(&v_free[(g - 1) & 1], ((g - 1) >> 1) & 1, wctl);
            {
              tc_fence_after();
              uint32_t o[HH];
              const uint32_t oc = tmem + t_lane + kColO + (item_n & 1) * HN + h0;
              if constexpr (HH == 32) tmem_ld_32x32b_x32(oc, o);
              else tmem_ld_32x32b_x16(oc, o);
              tmem_wait_ld();
#pragma unroll
              for (int i = 0; i < HH; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * aref[h0 + i]);
              if constexpr (HH == 32) tmem_st_32x32b_x32(oc, o);
              else tmem_st_32x32b_x16(oc, o);
              tmem_wait_st();
            }
          }
        }
        // P^T[c] is free once PV of tile g-2 is done.
        if (ok && g >= 2) ok = mbar_wait_abortable(&v_free[c], ((g >> 1) - 1) & 1, wctl);
        if (ok) {
          // P^T row of this token: heads 8i .. 8i+7 at i*2048 + tok*16 (MN-major B operand).
          uint8_t* dst = pt + c * L::kPTBytes + (h0 / 8) * 2048 + tok * 16;
          if (valid) {
            const uint64_t vs2 = f2(vs, vs);
#pragma unroll
            for (int h8 = 0; h8 < HH; h8 += 8) {
              uint32_t w[4];
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                const uint64_t pp = f2(ex2_approx(sv[h8 + 2 * e]), ex2_approx(sv[h8 + 2 * e + 1]));
                f2_split(f2_add(f2(l[h8 + 2 * e], l[h8 + 2 * e + 1]), pp), l[h8 + 2 * e], l[h8 + 2 * e + 1]);
                float q0, q1;
                f2_split(f2_mul(pp, vs2), q0, q1);
                w[e] = pack_f16x2(q0, q1);
              }
              *reinterpret_cast<uint4*>(dst + (h8 / 8) * 2048) = make_uint4(w[0], w[1], w[2], w[3]);
            }
          } else {
#pragma unroll
            for (int h8 = 0; h8 < HH; h8 += 8)
              *reinterpret_cast<uint4*>(dst + (h8 / 8) * 2048) = make_uint4(0u, 0u, 0u, 0u);
          }
        }
        fence_proxy_async_smem();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(&p_full[c]);
          mbar_arrive(&scale_free[ss]);
        }
      }
      // ---- end of item: per-head sums over the 128 tokens, then normalise O^T and write it.
      const int ob = item_n & 1;
      {
        float v[HH];
#pragma unroll
        for (int i = 0; i < HH; ++i) v[i] = l[i];
        const float ls = reduce_scatter<false, HH>(v, lane);
        if (lane < HH) lpart[quarter * HN + h0 + lane] = ls;
      }
      if (bar_red_or(kSoftBar, kSoftThreads, !ok)) break;
      // The item's G output rows and G log-sum-exps are contiguous in memory: both go
      // out as bulk copies from shared memory (O^T normalised into the P^T buffers,
      // which no MMA reads before this warpgroup writes the next item's first P^T;
      // the LSEs into the raise exchange, unused until then too).  The output is
      // 16-byte aligned (checked on the host); an LSE array that is not, or a row
      // of fewer than 4 LSEs, takes plain stores.
      const DecodeJob& jb = p.job[it.job];
      float* dst_o = it.direct ? jb.out + (job_row(jb, it.b) * Hq + it.kvh * G) * kHeadDim
                               : jb.ws_o + (((int64_t)it.b * jb.plan.max_splits + it.split) * Hq + it.kvh * G) * kHeadDim;
      float* dst_lse = it.direct ? (jb.lse_out ? jb.lse_out + job_row(jb, it.b) * Hq + it.kvh * G : nullptr)
                                 : jb.ws_lse + ((int64_t)it.b * jb.plan.max_splits + it.split) * Hq + it.kvh * G;
      const bool bulk_lse = dst_lse != nullptr && (reinterpret_cast<uintptr_t>(dst_lse) & 15u) == 0 && (G & 3) == 0;
      float* lse_stage = wmax;
      if (quarter == 0 && lane < HH) {
        const int h = h0 + lane;
        const float Ls = (lpart[h] + lpart[HN + h]) + (lpart[2 * HN + h] + lpart[3 * HN + h]);
        linv[h] = Ls > 0.0f ? 1.0f / Ls : 0.0f;
        if (h < G) {
          const float lse2 = Ls > 0.0f ? mref[h] + __log2f(Ls) : -INFINITY;
          const float lv = it.direct ? lse2 * kLn2 : lse2;  // the split merge works in log2 units
          if (bulk_lse) lse_stage[h] = lv;
          else if (dst_lse) dst_lse[h] = lv;
        }
      }
      named_barrier_sync(kSoftBar, kSoftThreads);
      ok = mbar_wait_abortable(&o_full[ob], (item_n >> 1) & 1, wctl);
      {
        tc_fence_after();
        uint32_t o[HH];
        const uint32_t oc = tmem + t_lane + kColO + ob * HN + h0;
        if constexpr (HH == 32) tmem_ld_32x32b_x32(oc, o);
        else tmem_ld_32x32b_x16(oc, o);
        tmem_wait_ld();
        float* stage = reinterpret_cast<float*>(pt);
#pragma unroll
        for (int i = 0; i < HH; ++i) stage[(h0 + i) * kHeadDim + tok] = __uint_as_float(o[i]) * linv[h0 + i];
      }
      tc_fence_before();
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(&o_empty[ob]);
      if (bar_red_or(kSoftBar, kSoftThreads, !ok)) break;
      if (sw == 0 && lane == 0) {
        bulk_s2g(dst_o, pt, (uint32_t)G * kHeadDim * 4);
        if (bulk_lse) bulk_s2g(dst_lse, lse_stage, (uint32_t)G * 4);
        bulk_commit();
      }
      ++item_n;
    }
    // The last bulk copies have landed before the CTA (and its shared memory) goes away.
    if (sw == 0 && lane == 0) bulk_wait_all();
  }

  tc_fence_before();
  __syncthreads();
  if (tid == 0 && *abort_flag) set_err(p.err, CAI_DEVERR_TIMEOUT);
  if (warp == 0) tmem_dealloc(tmem, kTmemCols);
  // A launch that did not wait for the kernel before it ends only after that kernel, so
  // that whatever follows in the stream finds both complete.
  if (p.overlap_prev) grid_dependency_wait();
}

// One warp per (sequence, head): merge the partial outputs of the splits by
// their log-sum-exp: out = sum_j 2^(lse_j - M) o_j / sum_j 2^(lse_j - M).
__global__ void __launch_bounds__(128) combine_kernel(const DecodeParams p, int job, int page_size) {
  grid_dependency_wait();
  grid_launch_dependents();
  const int gw = (int)((blockIdx.x * (int64_t)blockDim.x + threadIdx.x) >> 5);
  const int lane = threadIdx.x & 31;
  const int Hq = p.num_heads;
  if (gw >= p.batch * Hq) return;
  const int b = gw / Hq, h = gw - b * Hq;
  const DecodeJob& jb = p.job[job];
  int32_t L = p.ctx_len[b];
  if (jb.q_off) {  // a packed continuous batch: only its one-token rows were decoded
    const int32_t a = jb.q_off[b], e = jb.q_off[b + 1];
    if (!(a >= 0 && e == a + 1 && e <= jb.total_rows)) return;
    L = L + 1;
  }
  const SeqSplits sp = seq_splits(L, jb.window, jb.max_pages * page_size, jb.plan.chunk);
  if (!sp.valid || sp.nsplit <= 1) return;  // written by the decode kernel itself
  const int64_t orow = job_row(jb, b);
  static_assert(kMaxSplits <= 64, "two splits per lane");
  const int S = jb.plan.max_splits;        // <= 64: lane l holds splits l and l + 32
  const float* lse = jb.ws_lse + (int64_t)b * S * Hq + h;
  const float l0 = lane < sp.nsplit ? lse[(int64_t)lane * Hq] : -INFINITY;
  const float l1 = lane + 32 < sp.nsplit ? lse[(int64_t)(lane + 32) * Hq] : -INFINITY;
  float M = fmaxf(l0, l1);
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
  // Split weights 2^(lse_j - M), lane l holding those of splits l and l + 32.
  const float w0 = M == -INFINITY || lane >= sp.nsplit ? 0.0f : ex2_approx(l0 - M);
  const float w1 = M == -INFINITY || lane + 32 >= sp.nsplit ? 0.0f : ex2_approx(l1 - M);
  float wsum = w0 + w1;
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) wsum += __shfl_xor_sync(0xffffffffu, wsum, o);
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  const float4* rows = reinterpret_cast<const float4*>(jb.ws_o + ((int64_t)b * S * Hq + h) * kHeadDim) + lane;
  const int64_t stride = (int64_t)Hq * kHeadDim / 4;  // float4s from one split's row to the next
  // Four splits at a time so that their loads overlap.
  for (int j0 = 0; j0 < sp.nsplit; j0 += 4) {
    float4 o[4];
    float w[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int j = j0 + u;
      o[u] = j < sp.nsplit ? rows[j * stride] : make_float4(0.f, 0.f, 0.f, 0.f);
      const float wa = __shfl_sync(0xffffffffu, w0, j & 31), wb = __shfl_sync(0xffffffffu, w1, j & 31);
      w[u] = j < sp.nsplit ? (j < 32 ? wa : wb) : 0.0f;
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      acc.x = fmaf(w[u], o[u].x, acc.x);
      acc.y = fmaf(w[u], o[u].y, acc.y);
      acc.z = fmaf(w[u], o[u].z, acc.z);
      acc.w = fmaf(w[u], o[u].w, acc.w);
    }
  }
  const float inv = wsum > 0.0f ? 1.0f / wsum : 0.0f;
  reinterpret_cast<float4*>(jb.out + (orow * Hq + h) * kHeadDim)[lane] =
      make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv);
  if (jb.lse_out && lane == 0) jb.lse_out[orow * Hq + h] = wsum > 0.0f ? (M + __log2f(wsum)) * kLn2 : -INFINITY;
}

// The page pool as a 2-D tensor of 128-byte rows (a page of P tokens is
// page_bytes(P) / 128 consecutive rows: P K-code rows, P V-code rows, then the
// scale rows); one box is the 2P code rows of a page, landing 128-byte
// swizzled in shared memory.
bool encode_pool_map(CUtensorMap* map, const void* pages, int64_t num_pages, int P) {
  auto fn = tensor_map_encoder();
  if (!fn) return false;
  const int64_t rows = num_pages * (page_bytes(P) / 128);
  if (rows <= 0 || rows > 2147483647ll) return false;
  cuuint64_t dims[2] = {128, (cuuint64_t)rows};
  cuuint64_t strides[1] = {128};
  cuuint32_t box[2] = {128, (cuuint32_t)(2 * P)};
  cuuint32_t estr[2] = {1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(pages), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
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

template <int P, int HN>
cudaError_t launch_decode_ph(const DecodeParams& p, cudaStream_t stream) {
  static bool attr_set[64] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 64 && !attr_set[dev]) {
    // The register split inside the kernel assumes the launch register count.
    cudaFuncAttributes fa;
    cudaError_t e = cudaFuncGetAttributes(&fa, decode_kernel<P, HN>);
    if (e != cudaSuccess) return e;
    if (fa.numRegs != Roles<HN>::kRegsLaunch) return cudaErrorInvalidDeviceFunction;
    e = cudaFuncSetAttribute(decode_kernel<P, HN>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             Layout<HN>::kSmemBytes);
    if (e != cudaSuccess) return e;
    attr_set[dev] = true;
  }
  DecodeArgs a;
  a.p = p;
  for (int j = 0; j < p.num_slots; ++j)
    if (!encode_pool_map(&a.kv_map[j], p.pages[j], p.slot_pages[j], P)) return cudaErrorInvalidValue;
  const int64_t items = p.num_items;
  const int grid = (int)(items < num_sms() ? items : num_sms());
  cudaError_t e = launch_pdl(decode_kernel<P, HN>, dim3(grid), dim3(Roles<HN>::kThreads), Layout<HN>::kSmemBytes,
                             stream, a);
  for (int j = 0; e == cudaSuccess && j < p.num_jobs; ++j) {
    if (p.job[j].plan.max_splits <= 1) continue;
    const int64_t warps = (int64_t)p.batch * p.num_heads;
    e = launch_pdl(combine_kernel, dim3((unsigned)((warps + 3) / 4)), dim3(128), 0, stream, p, j, P);
  }
  return e;
}

template <int P>
cudaError_t launch_decode_p(const DecodeParams& p, cudaStream_t stream) {
  return p.num_heads / p.num_kv_heads <= 32 ? launch_decode_ph<P, 32>(p, stream) : launch_decode_ph<P, 64>(p, stream);
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
