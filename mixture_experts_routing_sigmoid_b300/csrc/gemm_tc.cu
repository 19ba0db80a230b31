// bf16 grouped GEMMs on the 5th-generation tensor cores (tcgen05 + TMEM + TMA), sm_103a.
//
//   MODE_GATE: u[t, e] = x[t] . W_g[e] + gate_bias[e]  (fp32 out; router linear layer,
//              "从零构建DeepSeekMoE", section 5.2)
//   MODE_UP:   h[r, j] = silu(A[r] . W13_p[j]) * (A[r] . W13_p[I + j])   (bf16 out)
//   MODE_DOWN: y[r, o] = h[r] . W2_p[o]                                   (bf16 out)
// Problem p < n_routed is expert p's segment (rows offsets[p] .. offsets[p+1]-1, read on the
// device); p == n_routed is the shared experts over all T tokens, with S shared experts
// stacked into one of intermediate size S*I ("DeepSeek MoE：从v1到v3的演进", DeepSeek-v1
// fine-grained experts and shared-expert isolation).
//
// Weight rows are the MMA's M side and tokens its N side ("swap AB"), and each tile runs on a
// pair of SMs (a cluster of two CTAs issuing tcgen05.mma.cta_group::2): D[w_row, token] =
// sum_k W[w_row, k] A[token, k]. Each CTA loads its own 128 weight rows and half of the tile's
// tokens; the pair's first CTA issues the MMA, which reads both CTAs' shared memory and writes
// each CTA's 128 rows of D into that CTA's TMEM. The instruction's N can be any multiple of
// 16, so a segment's ragged end costs at most 15 idle token columns instead of a mostly empty
// row tile, and in decode (a few tokens per expert) the weights stream through at full width
// while the token operand stays tiny.
//   UP:   per CTA, 64 intermediate features: its 128 weight rows interleave the gate and up
//         projections 16 rows at a time (rows 32q..32q+15 gate rows of features 16q..16q+15,
//         rows 32q+16..32q+31 the up rows of the same features; one 5-D TMA box loads them),
//         so warp q of the epilogue holds both halves of its 16 features and pairs them with
//         one shuffle before applying the SwiGLU in registers.
//   DOWN: 128 output features per CTA, up to 256 tokens per tile.
//   GATE: 128 router outputs per CTA (rows past n_routed read as zero), up to 256 tokens.
// A TMEM lane is one output feature and a column one token, so after tcgen05.ld a warp holds
// 32 consecutive features of each of 32 tokens: the epilogue stores straight from registers,
// each store instruction covering a contiguous run of one token's output row (neighbouring
// lanes swap values to write bf16 pairs). No shared-memory staging.
//
// Persistent kernel, one 352-thread CTA per SM. Tiles are numbered problem by problem (most
// rows first), weight tile by weight tile, token tile fastest (a segment's rows are split into
// equal token tiles). The first wave is one tile per CTA pair; after that a pair claims the next
// index from a counter when its producer starts the current tile (round robin without a
// counter), so the pairs sharing a weight tile run it together and its second read hits L2.
// (Claiming later, a few k blocks before the current tile's end, measured 1.5-3% slower.)
//   warp 0      TMA producer (both CTAs): this CTA's weight rows and token rows of one k block
//               per stage, in a 200 KB ring of stages sized by the tile (below). A k block is
//               128 elements, two 128-byte-swizzled units of 64, and each operand's two units
//               come in one TMA box (when K / 64 is odd the last block's second unit lies past
//               the end and reads as zeros). Two units per stage halve the barrier round trips
//               per FLOP against one-unit stages; one copy per operand and stage keeps the
//               producer's time per stage, which bounds how fast a tile with few tokens can
//               stream its weights, to about half of what a copy per unit and token box took.
//               Lane 0 alone walks a tile's stages. Completion of both CTAs' loads is counted
//               on the first CTA's full barrier; the MMA's commit frees the stage in both CTAs.
//   warp 1      TMEM owner (both CTAs) and, in the first CTA, MMA issuer: the whole warp waits
//               for each stage and computes its operands (so they are warp-uniform), and one
//               elected lane issues its tcgen05.mma (M=256, N=tile's tokens rounded up to 16,
//               K=16; four per unit) into one of two 256-column fp32 accumulators. (Issued from a
//               lone lane, a stage of eight MMAs took ~930 cycles of the issuer whatever N, the
//               bound of every tile with few tokens; warp-wide, decode T = 512 runs 2% faster.)
//   warps 2..9  epilogue (both CTAs): two warps per quarter of the TMEM lanes (a warp may only
//               read its own quarter), taking alternate 32-column chunks: tcgen05.ld, SwiGLU /
//               router bias, stores. Two warps per quarter keep a short tile's epilogue (a few
//               k blocks, as with the small intermediate sizes) shorter than the next tile's
//               main loop.
//   warp 10     tile scheduler: in the first CTA it claims, decodes and publishes each tile in
//               the CTA's local ring and sends it to the second CTA by st.async; in the second
//               CTA it relays the received tiles into that CTA's local ring.
// Token columns past the segment end belong to the next expert (or lie beyond the tensor,
// where TMA fills zeros); they are computed and never stored. Every mbarrier wait is bounded:
// on timeout the CTA raises an abort flag and the device error word, drains, frees TMEM and
// returns.
#include <cudaTypedefs.h>

#include "common.cuh"
#include "internal.h"

namespace moe {

namespace {

constexpr int BM = 128;                  // weight rows per CTA and operand (MMA M = 256)
constexpr int KU = 64;                   // reduction elements per unit (128 bytes of bf16)
constexpr int UNITS = 2;                 // units per stage (k block of 128 elements)
constexpr int MAXP = 258;
constexpr int MAXP4 = (MAXP + 3) & ~3;
constexpr int THREADS = 352;
constexpr int EPI_WARPS = 8;             // warps 2 .. 9
constexpr int SCHED_WARP = 10;
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t ACC_COLS = 256;       // two accumulators
constexpr int NTOKMAP = 3;               // token maps: boxes of 32, 64 or 128 rows
constexpr unsigned long long TIMEOUT_NS = 2000000000ull;    // 2 s per wait
constexpr unsigned long long GRACE_NS = 100000000ull;       // drain after an abort

constexpr int SQ = 4;                    // tile schedule ring slots
constexpr int kL2HintMaxTokens = 512;    // batches whose expert GEMMs use the L2 hints (measured:
                                         // 3-5% faster at 32 and 128 tokens; at 512 the combine
                                         // finds y in L2, 16.6 -> 14.2 us)
constexpr int A_UNIT = BM * KU * 2;      // this CTA's weight rows, one unit
constexpr int A_BYTES = UNITS * A_UNIT;

// Operand ring: RING_BYTES of shared memory cut into stages whose size follows the tile. A
// stage holds a k block of the CTA's 128 weight rows (32 KB) and of its half of the tile's
// tokens, so a tile with few tokens takes small stages and keeps more of them in flight:
// 256 tokens, 3 stages of 64 KB; 128 tokens, 4 of 48 KB; 64 or fewer, 5 of 34-40 KB. A tile
// with few tokens streams its weights and needs bytes in flight; a tile with many tokens needs
// the wide MMA; in a skewed batch both kinds run side by side in one launch, each at its depth.
// Stages are placed one after the other and wrap to the start of the ring when the next one
// does not fit; NS barrier pairs are used in turn, which also bounds the stages in flight.
// Launches whose tiles all stream many tokens (large batches) use NS = 3 (measured: rotating
// six slots there costs 1-2%); batches of at most kDeepRingMaxTokens tokens, where most
// tiles stream weights, use NS = NSLOT.
constexpr int TOK = 256;                 // tokens per tile at most (MMA N)
constexpr uint32_t RING_BYTES = 200 * 1024;
constexpr int NSLOT = 6;                 // more than the stages that fit at once
constexpr int kDeepRingMaxTokens = 512;
constexpr int kGateMaxSplits = 16;

// Every stage is filled by one weight copy and one token copy per CTA: the maps view K as
// (64-element unit, chunk of 64 units...) so that one box spans both k units of a stage (a TMA
// instruction costs the issuing thread on the order of a hundred cycles whatever its box, and
// the producer's per-stage time bounds the weight stream of a tile with few tokens).
struct TcParams {
  CUtensorMap tmW0, tmW1;    // weights: routed, shared (128 rows x 2 units; UP: interleaved 5-D)
  CUtensorMap tmX0[NTOKMAP]; // tokens, routed: 32, 64 or 128 rows x 2 units
  CUtensorMap tmX1[NTOKMAP]; // tokens, shared
  CUtensorMap tmXg;          // UP with row gather: x [T, H], box one row high (tile::gather4)
  const int32_t* row_token;  // UP with row gather: token of each routed row, else nullptr
  const int32_t* offsets;
  int rows_cap;              // rows of the routed activation and output tensors
  int n_routed, has_shared, T, H, I, S, N;
  void* out0;
  void* out1;
  const float* gate_bias;
  float* gate_part;          // GATE split-K: partial sums [splits][T][N]
  int* sched;                // tile counter (zero at launch) for the dynamic schedule, or null
  int l2_hints;              // 1: weights are streamed with evict_first, token rows loaded and
                             // outputs stored with evict_last (small batches: the weights pass
                             // through L2 once, the activations are read again soon)
  int splits, ku_per_split;  // GATE: K range split over `splits` tiles (1 = no split); units
                             // per split, even
  float* split_part;         // UP / DOWN tail split (see tail_split): partial accumulators, and
  int* split_cnt;            // arrival counters (zero at launch); nullptr: no tail split
  int offsets_early;         // 1: the offsets come from a kernel at least two launches back (the
                             // kernel ahead waited for it before letting this one start), so the
                             // tile schedule is built before waiting for the kernel ahead
  int* err;
};

// One tile, as decoded by the first CTA's producer and passed to every other role through the
// schedule rings (words only: it travels as three 16-byte vectors).
struct alignas(16) Tile {
  int prob;      // problem index; -1: no more tiles
  int f0;        // first output feature of the tile; this CTA's are f0 + feat_per_cta * rank ..
  int r0;        // first token row (in the problem's activation tensor)
  int nrows;     // token rows of this tile that are stored
  int ncols;     // MMA N: nrows rounded up to 16; each CTA holds ncols / 2 token rows
  int tok_rows;  // token rows per CTA and unit in a stage: 32, 64 or 128 (>= ncols / 2)
  int tsel;      // its token map: 0, 1, 2
  int ku0, ku;   // first k unit and k units (GATE split-K: this split's range)
  int kb;        // k blocks (stages): ku / UNITS rounded up
  int split;     // GATE split-K: which split. UP / DOWN: piece | pieces << 8 | split tile << 16
                 // for a piece of a tail tile (pieces >= 2), else 0
  int shared;    // the shared experts' problem
};
constexpr int TILE_WORDS = sizeof(Tile) / 4;
static_assert(TILE_WORDS == 12, "a tile travels as three 16-byte vectors");

struct SmemCtl {
  uint64_t full[NSLOT];        // first CTA's copy counts both CTAs' loads
  uint64_t empty[NSLOT];       // per CTA, arrived on by the MMA commit
  uint64_t tfull[2];           // per CTA, arrived on by the MMA commit
  uint64_t tempty[2];          // first CTA's copy: every epilogue warp of both CTAs
  uint64_t drain;
  // tile schedule: a CTA-local ring in each CTA (written by the CTA's producer, read by its
  // MMA issuer and epilogue warps) and a channel from the first CTA's producer to the second's
  uint64_t lfull[SQ];          // lsq[slot] holds the next tile
  uint64_t lempty[SQ];         // the slot's local readers are done with it
  uint64_t xfull[SQ];          // second CTA: xq[slot] arrived (tx-counted, 48 bytes)
  uint64_t xempty[SQ];         // first CTA: the second CTA's scheduler has read xq[slot]
  uint64_t took;               // first CTA: its producer has started the last published tile
  Tile lsq[SQ];
  Tile xq[SQ];
  int grow[SQ][TOK / 2];     // row gather: x row of each of this CTA's token rows of lsq[slot]
  uint32_t tmem_base;
  int abort_flag;
  int nprob;
  int total_tiles;            // work items: whole tiles, then the pieces of the split tail tiles
  int split_first;            // first split tile (== first piece's item)
  int split_s;                // pieces per split tile (0: no split)
  int tile_start[MAXP + 1];   // by position in `order`
  int order[MAXP];            // problems, most rows first (ties: lower index)
  alignas(16) uint32_t key[MAXP4];  // sort keys: rows high, reversed index low (0 past nprob)
  int chunk[THREADS / 32];    // per warp: its 32 positions' tile total
  int rows[MAXP];             // by problem: rows and first row of its segment
  int row0[MAXP];
};

constexpr size_t smem_bytes() { return (size_t)RING_BYTES + sizeof(SmemCtl); }
static_assert(smem_bytes() <= 232448, "shared memory budget of one CTA");

template <int MODE>
__device__ __forceinline__ int feat_total(const TcParams& p, bool shared) {
  if (MODE == MODE_UP) return shared ? p.S * p.I : p.I;
  if (MODE == MODE_DOWN) return p.H;
  return p.N;
}
// Output features of one CTA: UP 64 (gate and up rows of each), else 128.
template <int MODE>
__host__ __device__ constexpr int feat_per_cta() { return MODE == MODE_UP ? BM / 2 : BM; }
// Feature tiles of 2 * feat_per_cta outputs.
template <int MODE>
__device__ __forceinline__ int n_feat_tiles(const TcParams& p, bool shared) {
  return (feat_total<MODE>(p, shared) + 2 * feat_per_cta<MODE>() - 1) / (2 * feat_per_cta<MODE>());
}
template <int MODE>
__device__ __forceinline__ int k_units_of(const TcParams& p, bool shared) {
  if (MODE == MODE_DOWN) return (shared ? p.S * p.I : p.I) / KU;
  return p.H / KU;
}

template <int MODE>
__device__ __forceinline__ Tile decode_tile(const TcParams& p, const SmemCtl& c, int tile) {
  int lo = 0, hi = c.nprob - 1;  // largest q with tile_start[q] <= tile
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (c.tile_start[mid] <= tile) lo = mid; else hi = mid - 1;
  }
  Tile t;
  const int pos = lo;
  lo = c.order[pos];
  t.prob = lo;
  t.shared = (MODE != MODE_GATE) && lo >= p.n_routed;
  const int row0 = c.row0[lo], rows = c.rows[lo];
  const int ntt = (rows + TOK - 1) / TOK;
  int local = tile - c.tile_start[pos];
  t.split = 0;
  if (MODE == MODE_GATE && p.splits > 1) {  // split outermost
    const int per_split = ntt * n_feat_tiles<MODE>(p, false);
    t.split = local / per_split;
    local -= t.split * per_split;
  }
  const int ft = local / ntt;
  const int tt = local - ft * ntt;
  t.f0 = ft * 2 * feat_per_cta<MODE>();
  // a segment's rows split into ntt token tiles of equal size (a multiple of 16)
  const int per = (((rows + ntt - 1) / ntt) + 15) & ~15;
  t.r0 = row0 + tt * per;
  t.nrows = min(per, rows - tt * per);
  t.ncols = (t.nrows + 15) & ~15;
  const int half = t.ncols / 2;
  t.tsel = half <= 32 ? 0 : (half <= 64 ? 1 : 2);
  t.tok_rows = 32 << t.tsel;
  t.ku0 = 0;
  t.ku = k_units_of<MODE>(p, t.shared);
  if (MODE == MODE_GATE && p.splits > 1) {
    t.ku0 = t.split * p.ku_per_split;
    t.ku = min(p.ku_per_split, t.ku - t.ku0);
  }
  t.kb = (t.ku + UNITS - 1) / UNITS;
  return t;
}

// Checked build: a tile whose rows, features, k range or split fields leave their tensors (a
// corrupt schedule) is reported and its stores are skipped.
template <int MODE>
__device__ __forceinline__ bool tile_in_range(const TcParams& p, const Tile& t) {
  const int nprob = (MODE == MODE_GATE) ? 1 : p.n_routed + p.has_shared;
  const int rows = (MODE == MODE_GATE || t.shared) ? p.T : p.rows_cap;
  bool ok = t.prob >= 0 && t.prob < nprob && t.r0 >= 0 && t.nrows >= 1 && t.nrows <= TOK &&
            t.ncols >= t.nrows && t.ncols <= TOK && t.r0 + t.nrows <= rows && t.f0 >= 0 &&
            t.f0 < feat_total<MODE>(p, t.shared) && t.kb >= 1 && t.ku0 >= 0 &&
            t.ku0 + t.ku <= k_units_of<MODE>(p, t.shared);
  if (MODE == MODE_GATE) {
    ok = ok && t.split >= 0 && t.split < p.splits;
  } else {
    const int pieces = (t.split >> 8) & 0xff, piece = t.split & 0xff, sid = t.split >> 16;
    ok = ok && (pieces < 2 ? t.split == 0
                           : (piece < pieces && sid < kSplitMaxTiles &&
                              (sid + 1) * pieces <= kSplitMaxPieces));
  }
  return ok;
}

// Work item -> tile: items below split_first are whole tiles; the rest are the pieces of the
// split tiles, piece fastest, each a contiguous range of the tile's k blocks.
template <int MODE>
__device__ __forceinline__ Tile decode_item(const TcParams& p, const SmemCtl& c, int item) {
  const int S = c.split_s;
  if (MODE == MODE_GATE || S < 2 || item < c.split_first) return decode_tile<MODE>(p, c, item);
  const int j = item - c.split_first;
  const int sid = j / S, piece = j - sid * S;
  Tile t = decode_tile<MODE>(p, c, c.split_first + sid);
  const int lo = piece * t.kb / S, hi = (piece + 1) * t.kb / S;
  t.ku0 = lo * UNITS;
  t.ku = min(hi * UNITS, t.ku) - t.ku0;
  t.kb = hi - lo;
  t.split = piece | (S << 8) | (sid << 16);
  return t;
}

// Bytes of one unit of this CTA's token rows in a stage of tile t: the box rows it loads, or
// with the row gather its rows (a multiple of 8 rows: 1 KB aligned, as the 128-byte swizzle
// wants).
__device__ __forceinline__ uint32_t tok_unit_bytes(const Tile& t, bool gathered) {
  if (gathered) return (uint32_t)(t.ncols / 2) * KU * 2;
  return (uint32_t)t.tok_rows * KU * 2;
}
__device__ __forceinline__ uint32_t stage_bytes_of(const Tile& t, bool gathered) {
  return A_BYTES + UNITS * tok_unit_bytes(t, gathered);
}
// Placement of consecutive stages in the ring: each after the previous one, or at the start
// when it would run past the end. Producer and MMA issuer of both CTAs walk the same sequence of
// tiles and so place every stage at the same offset.
struct RingPlace {
  uint32_t next = 0;
  __device__ __forceinline__ uint32_t place(uint32_t bytes) {
    const uint32_t off = next + bytes > RING_BYTES ? 0u : next;
    next = off + bytes;
    return off;
  }
};

// Tail split: W whole tiles on P CTA pairs end in a wave of R = W mod P tiles (all W when
// W < P) that leaves P - R pairs idle. When R <= P / 2, each of those R tiles is cut along K
// into S = P / R pieces (at most 8, and at least kSplitMinBlocks k blocks of a routed tile
// each: a piece pays its own ring fill and partial round trip), which run as the last work
// items. Sets first = W - R and pieces = S, or pieces = 0 (no split). Only the up projection
// splits: its tiles run over the hidden size (56 k blocks at 7168); the down projection's run
// over one expert's intermediate size, and measured at 2048 (16 k blocks, two pieces) the
// pieces' ring fills cost more than the shorter wave saves.
constexpr int kSplitMinBlocks = 8;
__device__ __forceinline__ void tail_split(int W, int P, int kb_routed, int& first, int& pieces) {
  first = W;
  pieces = 0;
  if (W <= 0 || P <= 1) return;
  const int R = W % P;
  if (R == 0 || 2 * R > P || R > kSplitMaxTiles) return;
  int S = P / R;
  S = min(S, 8);
  S = min(S, kb_routed / kSplitMinBlocks);
  S = min(S, kSplitMaxPieces / R);
  if (S < 2) return;
  first = W - R;
  pieces = S;
}

__device__ __forceinline__ Tile end_tile() {
  Tile t;
  int* w = reinterpret_cast<int*>(&t);
#pragma unroll
  for (int i = 0; i < TILE_WORDS; ++i) w[i] = 0;
  t.prob = -1;
  return t;
}

// This CTA's copies for tile t, fixed along K: the weight map and box (UP: 5-D coordinates
// (0, 0, wa = 2 * expert, wb = first 16-feature group, chunk); else 3-D (0, wa = row, chunk))
// and the token map and first row (3-D (0, trow, chunk)). The chunk coordinate is the stage's
// first k unit; one box brings that unit and the next.
struct TileBoxes {
  const CUtensorMap* tw;
  const CUtensorMap* tx;
  int wa, wb, trow;
};

template <int MODE>
__device__ __forceinline__ TileBoxes tile_boxes(const TcParams& p, const Tile& t, uint32_t rank) {
  TileBoxes b;
  b.tw = t.shared ? &p.tmW1 : &p.tmW0;
  b.tx = t.shared ? &p.tmX1[t.tsel] : &p.tmX0[t.tsel];
  int fc = t.f0 + (int)rank * feat_per_cta<MODE>();    // this CTA's first feature
  if (fc >= feat_total<MODE>(p, t.shared)) fc = t.f0;  // past the end: recompute CTA 0's rows
  b.wb = 0;
  if (MODE == MODE_UP) {
    const int s = fc / p.I, j = fc - s * p.I;          // expert (shared: stacked), feature in it
    b.wa = 2 * (t.shared ? s : t.prob);
    b.wb = j / 16;
  } else if (MODE == MODE_DOWN) {
    // shared: the k range runs over the shared experts' stacked intermediate sizes; the
    // stage's expert adds its H rows (see the producer)
    b.wa = t.shared ? fc : t.prob * p.H + fc;
  } else {
    b.wa = fc;
  }
  b.trow = t.r0 + (int)rank * (t.ncols / 2);
  return b;
}

__device__ __forceinline__ void grace_wait(uint32_t bar, uint32_t parity) {
  const unsigned long long t0 = globaltimer_ns();
  while (!mbar_try_wait(bar, parity))
    if (globaltimer_ns() - t0 > GRACE_NS) break;
}

__device__ __forceinline__ void grace_sleep() {
  const unsigned long long t0 = globaltimer_ns();
  while (globaltimer_ns() - t0 < GRACE_NS / 10) {
  }
}

__device__ __forceinline__ float silu_mul(float g, float u) {
  return g / (1.0f + __expf(-g)) * u;
}

// Stores this lane's feature f (f of lanes l and l^1 differ in the last bit) for tokens
// row0 .. row0 + NT - 1 of a row-major bf16 output with leading dimension ld: lanes l and l^1
// swap one value per token pair so that the even lane writes features (f, f+1) of the even
// token and the odd lane features (f-1, f) of the odd token, 4 bytes each.
template <int NT>
__device__ __forceinline__ void store_bf16_chunk(const float (&v)[NT], __nv_bfloat16* out,
                                                 size_t ld, size_t row0, int nvalid, int f,
                                                 bool fvalid, int lane, bool hint,
                                                 uint64_t policy) {
  const bool odd = lane & 1;
  __nv_bfloat16* base = out + row0 * ld + (odd ? f - 1 : f);
#pragma unroll
  for (int i = 0; i < NT; i += 2) {
    const float mine = odd ? v[i] : v[i + 1];
    const float other = __shfl_xor_sync(FULL_MASK, mine, 1);
    const int tok = odd ? i + 1 : i;
    const uint32_t pk = odd ? pack_bf16x2(other, v[i + 1]) : pack_bf16x2(v[i], other);
    if (fvalid && tok < nvalid) {
      if (hint) st_u32_hint(base + (size_t)tok * ld, pk, policy);
      else *reinterpret_cast<uint32_t*>(base + (size_t)tok * ld) = pk;
    }
  }
}

// ---- tile schedule: the first CTA's scheduler warp decides which tile the pair takes next,
// decodes it and publishes it in its CTA's local ring and, with asynchronous remote stores that
// count on a barrier of the second CTA (st.async), to the second CTA's scheduler warp, which
// republishes it in its own local ring. The producer, MMA issuer and epilogue warps only read
// their local ring: no wait on their path is cluster-scope, and no decoding sits between two
// stages of a producer or MMA issuer.
constexpr uint32_t LOCAL_READERS_0 = 2 + EPI_WARPS;  // first CTA: producer, MMA issuer, epilogue
constexpr uint32_t LOCAL_READERS_1 = 1 + EPI_WARPS;  // second CTA: producer, epilogue
constexpr uint32_t TILE_BYTES = sizeof(Tile);

__device__ __forceinline__ void sts_tile(uint32_t a, const Tile& t) {
  const int* w = reinterpret_cast<const int*>(&t);
#pragma unroll
  for (int i = 0; i < TILE_WORDS; i += 4)
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};"
                 :: "r"(a + 4 * i), "r"(w[i]), "r"(w[i + 1]), "r"(w[i + 2]), "r"(w[i + 3]) : "memory");
}
__device__ __forceinline__ void lds_tile(uint32_t a, Tile& t) {
  int* w = reinterpret_cast<int*>(&t);
#pragma unroll
  for (int i = 0; i < TILE_WORDS; i += 4)
    asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(w[i]), "=r"(w[i + 1]), "=r"(w[i + 2]), "=r"(w[i + 3]) : "r"(a + 4 * i) : "memory");
}

// Row gather: the x row of each of this CTA's token rows of tile t (rows t.r0 + rank * ncols/2
// ..), into slot qs's row list. Rows past the tile's stored rows (MMA padding, never stored)
// take the tile's first token. Warp-wide.
__device__ __forceinline__ void fill_rows(SmemCtl& c, uint32_t qs, const TcParams& p,
                                          const Tile& t, uint32_t rank) {
  const int half = t.ncols / 2;
  const int base = t.r0 + (int)rank * half;
  const int end = t.r0 + t.nrows;
  const int pad = __ldg(p.row_token + t.r0);
  for (int i = threadIdx.x & 31; i < half; i += 32) {
    const int r = base + i;
    const int tok = r < end ? __ldg(p.row_token + r) : pad;
    if (kChecks && (tok < 0 || tok >= p.T)) set_error(p.err, ERR_DEVICE_CHECK);
    c.grow[qs][i] = min(max(tok, 0), p.T - 1);
  }
  __threadfence_block();
  __syncwarp();
}

// Publish `t` in slot `qs` of this CTA's local ring (with its gathered rows when gp is given).
// Warp-wide (scheduler warp).
__device__ __forceinline__ bool ring_publish(SmemCtl& c, uint32_t qs, uint32_t qph, const Tile& t,
                                             volatile int* abort_flag, int* err,
                                             const TcParams* gp = nullptr, uint32_t rank = 0) {
  if (!warp_wait_bounded(smem_u32(&c.lempty[qs]), qph ^ 1u, abort_flag, err, TIMEOUT_NS))
    return false;
  if (gp != nullptr && t.prob >= 0 && !t.shared) fill_rows(c, qs, *gp, t, rank);
  if ((threadIdx.x & 31) == 0) {
    sts_tile(smem_u32(&c.lsq[qs]), t);
    mbar_arrive(smem_u32(&c.lfull[qs]));
  }
  __syncwarp();
  return true;
}

// First CTA: send `t` to slot `qs` of the second CTA's channel. Warp-wide (scheduler warp).
__device__ __forceinline__ bool ring_send(SmemCtl& c, uint32_t qs, uint32_t qph, const Tile& t,
                                          volatile int* abort_flag, int* err) {
  if (!warp_wait_bounded(smem_u32(&c.xempty[qs]), qph ^ 1u, abort_flag, err, TIMEOUT_NS))
    return false;
  if ((threadIdx.x & 31) == 0) {
    const int* w = reinterpret_cast<const int*>(&t);
    const uint32_t dst = mapa_shared(smem_u32(&c.xq[qs]), 1);
    const uint32_t rb = mapa_shared(smem_u32(&c.xfull[qs]), 1);
#pragma unroll
    for (int i = 0; i < TILE_WORDS; i += 4)
      asm volatile(
          "st.async.shared::cluster.mbarrier::complete_tx::bytes.v4.b32 [%0], {%1, %2, %3, %4}, [%5];"
          :: "r"(dst + 4 * i), "r"(w[i]), "r"(w[i + 1]), "r"(w[i + 2]), "r"(w[i + 3]), "r"(rb)
          : "memory");
  }
  __syncwarp();
  return true;
}

// Second CTA: receive slot `qs` of the channel (warp-wide), re-arm its barrier for the next
// use and hand the slot back to the first CTA.
__device__ __forceinline__ bool ring_recv(SmemCtl& c, uint32_t qs, uint32_t qph, Tile& t,
                                          volatile int* abort_flag, int* err) {
  if (!warp_wait_bounded(smem_u32(&c.xfull[qs]), qph, abort_flag, err, TIMEOUT_NS)) return false;
  lds_tile(smem_u32(&c.xq[qs]), t);
  __syncwarp();
  if ((threadIdx.x & 31) == 0) {
    mbar_expect_tx(smem_u32(&c.xfull[qs]), TILE_BYTES);
    // the tile is in registers (the arrive takes a word of it as an operand), so a relaxed
    // arrive cannot overtake the reads
    asm volatile("mbarrier.arrive.relaxed.cluster.shared::cluster.b64 _, [%0];"
                 :: "r"(mapa_shared(smem_u32(&c.xempty[qs]), 0)), "r"(t.prob) : "memory");
  }
  return true;
}

// Warp-wide ring_take: lane 0 waits, every lane reads the slot, lane 0 releases it.
__device__ __forceinline__ bool ring_take_warp(SmemCtl& c, uint32_t qs, uint32_t qph, Tile& t,
                                               volatile int* abort_flag, int* err) {
  if (!warp_wait_bounded(smem_u32(&c.lfull[qs]), qph, abort_flag, err, TIMEOUT_NS)) return false;
  lds_tile(smem_u32(&c.lsq[qs]), t);
  __syncwarp();
  if ((threadIdx.x & 31) == 0) mbar_arrive(smem_u32(&c.lempty[qs]));
  return true;
}

template <int MODE, int NS>
__global__ void __launch_bounds__(THREADS, 1) tc_gemm_kernel(const __grid_constant__ TcParams p) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  const uint32_t sbase = smem_u32(smem_raw);  // 128-byte swizzle atoms want 1 KB alignment
  uint8_t* sgen = smem_raw;
  if (sbase & 1023u) {  // not expected: report it instead of computing with a wrong layout
    if (threadIdx.x == 0) set_error(p.err, ERR_DEVICE_CHECK);
    return;
  }
  SmemCtl& c = *reinterpret_cast<SmemCtl*>(sgen + RING_BYTES);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();   // 0: issues the MMA; 1: its peer
  const int pair = blockIdx.x >> 1, npairs = gridDim.x >> 1;

  auto bar = [](const uint64_t& b) { return smem_u32(&b); };

  if (threadIdx.x == 0) {
    for (int s = 0; s < NSLOT; ++s) { mbar_init(bar(c.full[s]), 1); mbar_init(bar(c.empty[s]), 1); }
    for (int a = 0; a < 2; ++a) {
      mbar_init(bar(c.tfull[a]), 1);
      mbar_init(bar(c.tempty[a]), 2 * EPI_WARPS);  // every epilogue warp of both CTAs
    }
    mbar_init(bar(c.drain), 1);
    for (int s = 0; s < SQ; ++s) {
      mbar_init(bar(c.lfull[s]), 1);
      mbar_init(bar(c.lempty[s]), rank == 0 ? LOCAL_READERS_0 : LOCAL_READERS_1);
      mbar_init(bar(c.xfull[s]), 1);
      mbar_init(bar(c.xempty[s]), 1);
    }
    mbar_init(bar(c.took), 1);
    // the channel's first phases: one arrival (this one) and the tile's bytes
    if (rank == 1)
      for (int s = 0; s < SQ; ++s) mbar_expect_tx(bar(c.xfull[s]), TILE_BYTES);
    c.abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) tmem_alloc_pair(smem_u32(&c.tmem_base), TMEM_COLS);

  // The kernel ahead in the stream has finished and its writes are visible after pdl_wait.
  // The schedule below reads only the segment offsets; when they come from further back
  // (offsets_early) it is built first, overlapping the end of the kernel ahead.
  const bool early = MODE != MODE_GATE && p.offsets_early != 0;
  if (!early) {
    pdl_wait();
    pdl_trigger();
  }
  // ---- problems in order of decreasing rows, so that the longest run first and the pairs
  // finish together; then the tile prefix over that order (counts depend on device offsets)
  const int nprob = (MODE == MODE_GATE) ? 1 : p.n_routed + p.has_shared;
  for (int q = threadIdx.x; q < MAXP4; q += THREADS) {
    if (q >= nprob) {
      c.key[q] = 0u;  // below every problem's key
      continue;
    }
    int rows = p.T, row0 = 0;
    if (MODE != MODE_GATE && q < p.n_routed) {
      row0 = __ldcg(p.offsets + q);
      const int end = __ldcg(p.offsets + q + 1);
      rows = max(end - row0, 0);
      if (kChecks && (row0 < 0 || end < row0 || end > p.rows_cap)) {
        set_error(p.err, ERR_DEVICE_CHECK);  // a segment outside the rows: skip the problem
        row0 = 0;
        rows = 0;
      }
    }
    c.rows[q] = rows;
    c.row0[q] = row0;
    // distinct keys (the reversed index in the low bits): the ranks are a permutation
    c.key[q] = (uint32_t)min(rows, (1 << 22) - 1) << 9 | (uint32_t)(511 - q);
  }
  __syncthreads();
  for (int q = threadIdx.x; q < nprob; q += THREADS) {
    const uint32_t kq = c.key[q];
    int rank = 0;
#pragma unroll 8
    for (int o = 0; o < nprob; o += 4) {  // four keys per shared load, loads overlapped
      const uint4 k4 = *reinterpret_cast<const uint4*>(&c.key[o]);
      rank += (k4.x > kq) + (k4.y > kq) + (k4.z > kq) + (k4.w > kq);
    }
    c.order[rank] = q;
  }
  __syncthreads();
  // tile prefix over the order: thread i counts position i's tiles; warp scans, then the warp
  // totals (nprob <= MAXP < THREADS, so one pass)
  int cnt = 0, incl = 0;
  {
    const int i = threadIdx.x;
    if (i < nprob) {
      const int q = c.order[i];
      const bool sh = (MODE != MODE_GATE) && q >= p.n_routed;
      cnt = ((c.rows[q] + TOK - 1) / TOK) * n_feat_tiles<MODE>(p, sh);
      if (MODE == MODE_GATE) cnt *= p.splits;
    }
    incl = cnt;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int v = __shfl_up_sync(FULL_MASK, incl, o);
      if (lane >= o) incl += v;
    }
    if (lane == 31) c.chunk[warp] = incl;
  }
  __syncthreads();
  {
    const int i = threadIdx.x;
    int before = 0;
    for (int w = 0; w < warp; ++w) before += c.chunk[w];
    if (i < nprob) c.tile_start[i] = before + incl - cnt;
    if (i == THREADS - 1) {  // the last thread: every warp's total is before it or its own
      const int run = before + incl;
      c.tile_start[nprob] = run;
      c.nprob = nprob;
      int first = run, pieces = 0;
      if (MODE == MODE_UP && p.split_part != nullptr && p.split_cnt != nullptr)
        tail_split(run, (int)(gridDim.x >> 1), (k_units_of<MODE>(p, false) + UNITS - 1) / UNITS,
                   first, pieces);
      c.split_first = first;
      c.split_s = pieces;
      c.total_tiles = first + (run - first) * (pieces > 1 ? pieces : 1);
    }
  }
  // both CTAs' barriers are initialised before either CTA signals the other's
  tc_fence_before();
  __syncthreads();
  cluster_sync();
  tc_fence_after();
  if (early) {
    pdl_wait();
    pdl_trigger();
  }
  const uint32_t tmem_base = c.tmem_base;
  const int total = c.total_tiles;
  volatile int* abort_flag = &c.abort_flag;

  if (warp == 0) {
    // ================================================================ TMA producer
    // Lane 0 alone: no warp-wide step between two stages (a shuffle or warp barrier there
    // costs the stream of a tile with few tokens more than its copies do).
    if (lane == 0) {
      const bool gather = MODE == MODE_UP && p.row_token != nullptr;
      tma_prefetch_desc(&p.tmW0);
      if (gather) {
        tma_prefetch_desc(&p.tmXg);
      } else {
#pragma unroll
        for (int i = 0; i < NTOKMAP; ++i) tma_prefetch_desc(&p.tmX0[i]);
      }
      if (MODE != MODE_GATE && p.has_shared) {
        tma_prefetch_desc(&p.tmW1);
#pragma unroll
        for (int i = 0; i < NTOKMAP; ++i) tma_prefetch_desc(&p.tmX1[i]);
      }
      const bool hint = p.l2_hints != 0;
      const uint64_t pol_w = l2_policy_evict_first(), pol_x = l2_policy_evict_last();
      uint32_t seq = 0;                           // stages issued so far
      RingPlace place;
      uint32_t hlo[NS - 1], hhi[NS - 1];          // ring bytes of stages seq-1, seq-2, ...
#pragma unroll
      for (int i = 0; i < NS - 1; ++i) hlo[i] = hhi[i] = 0;
      uint32_t issued_mask = 0, last_parity = 0;  // per slot: issued at least once / its parity
      uint32_t qs = 0, qph = 0;                   // schedule ring slot and phase
      bool ok = true;
      // Places stage `seq` (`bytes` long) and waits for the release of the stage it must
      // follow: the latest earlier stage whose bytes it overlaps, or the barrier slot's previous
      // stage (the MMA commits stages in order, so that one release covers every earlier one).
      auto place_and_wait = [&](uint32_t bytes, uint32_t& off, uint32_t& slot) -> bool {
        off = place.place(bytes);
        int w = (int)seq - NS;
#pragma unroll
        for (int i = 0; i < NS - 1; ++i) {
          const int j = (int)seq - 1 - i;
          if (j > w && off < hhi[i] && hlo[i] < off + bytes) w = j;
        }
#pragma unroll
        for (int i = NS - 2; i > 0; --i) { hlo[i] = hlo[i - 1]; hhi[i] = hhi[i - 1]; }
        hlo[0] = off;
        hhi[0] = off + bytes;
        slot = seq % NS;
        if (w < 0) return true;
        return mbar_wait_bounded(bar(c.empty[(uint32_t)w % NS]), ((uint32_t)w / NS) & 1u,
                                 abort_flag, p.err, TIMEOUT_NS);
      };
      auto issued = [&](uint32_t slot) {
        issued_mask |= 1u << slot;
        last_parity = (last_parity & ~(1u << slot)) | (((seq / NS) & 1u) << slot);
        ++seq;
      };
      while (ok) {
        if (!mbar_wait_bounded(smem_u32(&c.lfull[qs]), qph, abort_flag, p.err, TIMEOUT_NS)) {
          ok = false;
          break;
        }
        Tile t;
        lds_tile(smem_u32(&c.lsq[qs]), t);
        const uint32_t tq = qs;  // the slot (and its row list) stays held until the tile is issued
        if (++qs == SQ) { qs = 0; qph ^= 1u; }
        if (t.prob < 0) {
          mbar_arrive(smem_u32(&c.lempty[tq]));
          break;
        }
        if (rank == 0) mbar_arrive(bar(c.took));  // the scheduler may claim the next tile
        const TileBoxes b = tile_boxes<MODE>(p, t, rank);
        if (gather && !t.shared) {
          // routed rows gathered from x: the weight box, then one gather4 per four of this
          // CTA's token rows and unit
          const int half = t.ncols / 2;
          const uint32_t tok_bytes = tok_unit_bytes(t, true);
          const uint32_t sbytes = stage_bytes_of(t, true);
          const int4* grow = reinterpret_cast<const int4*>(&c.grow[tq][0]);
          for (int kb = 0; kb < t.kb; ++kb) {
            const int nu = min(UNITS, t.ku - kb * UNITS);
            const int kc = t.ku0 + kb * UNITS;
            // the weight box always brings both units (past the end of K: zeros)
            const uint32_t tx = 2 * (A_BYTES + nu * tok_bytes);
            uint32_t off, slot;
            if (!place_and_wait(sbytes, off, slot)) {
              ok = false;
              break;
            }
            const uint32_t fb = mapa_shared(bar(c.full[slot]), 0);
            const uint32_t sa = sbase + off;
            if (rank == 0) mbar_expect_tx(bar(c.full[slot]), tx);
            if (hint) tma_load_5d_pair_hint(sa, b.tw, fb, 0, 0, b.wa, b.wb, kc, pol_w);
            else tma_load_5d_pair(sa, b.tw, fb, 0, 0, b.wa, b.wb, kc);
            for (int i = 0; 4 * i < half; ++i) {
              const int4 r = grow[i];
              const uint32_t sg = sa + A_BYTES + i * (4 * KU * 2);
              tma_gather4_pair(sg, &p.tmXg, fb, kc * KU, r.x, r.y, r.z, r.w);
              if (nu > 1)
                tma_gather4_pair(sg + tok_bytes, &p.tmXg, fb, (kc + 1) * KU, r.x, r.y, r.z, r.w);
            }
            issued(slot);
          }
        } else {
          // Every copy brings both units of the stage (past the end of K: zeros), so each stage
          // expects its full size.
          const uint32_t sbytes = stage_bytes_of(t, false);
          const uint32_t tx = 2 * sbytes;
          // shared down projection: (ws, wkc) = the shared expert of the stage's first unit
          // and the unit within its intermediate size (a multiple of 128: no stage straddles
          // two experts)
          const bool stacked = MODE == MODE_DOWN && t.shared;
          const int ipu = stacked ? p.I / KU : 0;
          int ws = stacked ? t.ku0 / ipu : 0;
          int wkc = stacked ? t.ku0 - ws * ipu : t.ku0;
          for (int kb = 0; kb < t.kb; ++kb) {
            const int kc = t.ku0 + kb * UNITS;
            const int wrow = b.wa + ws * p.H;
            uint32_t off, slot;
            if (!place_and_wait(sbytes, off, slot)) {
              ok = false;
              break;
            }
            const uint32_t fb = mapa_shared(bar(c.full[slot]), 0);  // the first CTA's barrier
            const uint32_t sa = sbase + off;
            const uint32_t sb = sa + A_BYTES;
            if (rank == 0) mbar_expect_tx(bar(c.full[slot]), tx);
            if (MODE == MODE_UP) {
              if (hint) tma_load_5d_pair_hint(sa, b.tw, fb, 0, 0, b.wa, b.wb, wkc, pol_w);
              else tma_load_5d_pair(sa, b.tw, fb, 0, 0, b.wa, b.wb, wkc);
            } else {
              if (hint) tma_load_3d_pair_hint(sa, b.tw, fb, 0, wrow, wkc, pol_w);
              else tma_load_3d_pair(sa, b.tw, fb, 0, wrow, wkc);
            }
            if (hint) tma_load_3d_pair_hint(sb, b.tx, fb, 0, b.trow, kc, pol_x);
            else tma_load_3d_pair(sb, b.tx, fb, 0, b.trow, kc);
            issued(slot);
            wkc += UNITS;
            if (stacked && wkc >= ipu) {
              wkc -= ipu;
              ++ws;
            }
          }
        }
        mbar_arrive(smem_u32(&c.lempty[tq]));
      }
      if (ok && seq > 0) {
        // tail: wait until the MMA has released the last stage (and with it every earlier one)
        const uint32_t w = seq - 1;
        mbar_wait_bounded(bar(c.empty[w % NS]), (w / NS) & 1u, abort_flag, p.err, TIMEOUT_NS);
      }
      if (*abort_flag) {
        if (rank == 0) {
          for (int s = 0; s < NS; ++s)
            if ((issued_mask >> s) & 1u) grace_wait(bar(c.full[s]), (last_parity >> s) & 1u);
        } else {
          grace_sleep();  // this CTA's loads complete on the other CTA's barriers
        }
      }
    }
  } else if (warp == 1) {
    // ================================================================ MMA issuer (first CTA)
    // The whole warp walks the tiles and stages and computes every operand (so the operands are
    // warp-uniform); one elected lane issues the MMAs and commits.
    if (rank == 0) {
      const bool leader = elect_one_sync();
      uint32_t slot = 0, sphase = 0, acc = 0, aphase = 0, qs = 0, qph = 0;
      RingPlace place;
      bool ok = true;
      while (ok) {
        Tile t;
        if (!ring_take_warp(c, qs, qph, t, abort_flag, p.err)) break;
        if (++qs == SQ) { qs = 0; qph ^= 1u; }
        if (t.prob < 0) break;
        const uint32_t idesc = idesc_bf16_f32(2 * BM, t.ncols);
        const bool gathered = MODE == MODE_UP && p.row_token != nullptr && !t.shared;
        const uint32_t tok_bytes = tok_unit_bytes(t, gathered);
        const uint32_t sbytes = stage_bytes_of(t, gathered);
        if (!warp_wait_bounded(bar(c.tempty[acc]), aphase ^ 1u, abort_flag, p.err, TIMEOUT_NS)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + acc * ACC_COLS;
        for (int kb = 0; kb < t.kb; ++kb) {
          // the stage's descriptors are ready before its data: nothing but the MMAs follows
          // the wait
          const uint32_t sa = sbase + place.place(sbytes);
          const uint64_t ad0 = sdesc_k_sw128(sa), bd0 = sdesc_k_sw128(sa + A_BYTES);
          const uint64_t ad1 = ad0 + (A_UNIT >> 4), bd1 = bd0 + (tok_bytes >> 4);
          const bool two = t.ku - kb * UNITS > 1;
          const uint32_t acc0 = kb > 0 ? 1u : 0u;
          ready_before(ad0); ready_before(bd0); ready_before(ad1); ready_before(bd1);
          // every lane polls the barrier; the warp goes on only if all lanes saw the phase end
          const bool got = mbar_wait_bounded(bar(c.full[slot]), sphase, abort_flag, p.err,
                                             TIMEOUT_NS);
          if (!__all_sync(FULL_MASK, got)) {
            ok = false;
            break;
          }
          tc_fence_after();
          if (leader) {
#pragma unroll
            for (int kk = 0; kk < KU / 16; ++kk)
              tc_mma_f16_pair(d_tmem, ad0 + 2u * kk, bd0 + 2u * kk, idesc, kk > 0 ? 1u : acc0);
            if (two) {
#pragma unroll
              for (int kk = 0; kk < KU / 16; ++kk)
                tc_mma_f16_pair(d_tmem, ad1 + 2u * kk, bd1 + 2u * kk, idesc, 1u);
            }
            tc_commit_pair_mc(bar(c.empty[slot]), 0x3);
          }
          __syncwarp();
          if (++slot == NS) { slot = 0; sphase ^= 1u; }
        }
        if (!ok) break;
        if (leader) tc_commit_pair_mc(bar(c.tfull[acc]), 0x3);
        __syncwarp();
        acc ^= 1u;
        if (acc == 0) aphase ^= 1u;
      }
      if (*abort_flag && leader) {
        tc_commit_pair_mc(bar(c.drain), 0x1);  // arrives once every MMA issued above completed
        grace_wait(bar(c.drain), 0);
      }
      __syncwarp();
    }
  } else if (warp == SCHED_WARP) {
    // ================================================================ tile scheduler
    // First CTA: tiles one per pair in pair order first; then either round robin (static) or,
    // with a tile counter, in index order to whichever pair asks next: a pair claims its next
    // tile when its producer starts the current one, so the pairs that share a weight tile start
    // it within about a microsecond of each other and its second read hits L2. Each tile is
    // decoded once here. Second CTA: relays the first CTA's tiles into its local ring.
    uint32_t qs = 0, qph = 0, tph = 0;
    int cur = pair;
    for (;;) {
      Tile t;
      const TcParams* gp = (MODE == MODE_UP && p.row_token != nullptr) ? &p : nullptr;
      if (rank == 0) {
        t = cur < total ? decode_item<MODE>(p, c, cur) : end_tile();
        if (!ring_publish(c, qs, qph, t, abort_flag, p.err, gp, rank) ||
            !ring_send(c, qs, qph, t, abort_flag, p.err))
          break;
      } else {
        if (!ring_recv(c, qs, qph, t, abort_flag, p.err) ||
            !ring_publish(c, qs, qph, t, abort_flag, p.err, gp, rank))
          break;
      }
      if (++qs == SQ) { qs = 0; qph ^= 1u; }
      if (t.prob < 0) break;
      if (rank == 0) {
        if (!warp_wait_bounded(bar(c.took), tph, abort_flag, p.err, TIMEOUT_NS)) break;
        tph ^= 1u;
        if (lane == 0) cur = p.sched != nullptr ? npairs + atomicAdd(p.sched, 1) : cur + npairs;
        cur = __shfl_sync(FULL_MASK, cur, 0);
      }
    }
  } else {
    // ================================================================ epilogue
    const int q = warp & 3;               // TMEM lane quarter this warp may access
    const int h = (warp - 2) >> 2;        // chunks ch with ch % 2 == h
    const bool hint = p.l2_hints != 0;
    const uint64_t pol_o = l2_policy_evict_last();
    const uint32_t tempty0 = mapa_shared(bar(c.tempty[0]), 0);
    const uint32_t tempty1 = mapa_shared(bar(c.tempty[1]), 0);
    uint32_t acc = 0, aphase = 0, qs = 0, qph = 0;
    for (;;) {
      Tile t;
      if (!ring_take_warp(c, qs, qph, t, abort_flag, p.err)) break;
      if (++qs == SQ) { qs = 0; qph ^= 1u; }
      if (t.prob < 0) break;
      if (!warp_wait_bounded(bar(c.tfull[acc]), aphase, abort_flag, p.err, TIMEOUT_NS)) break;
      tc_fence_after();
      const uint32_t tb = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + acc * ACC_COLS;
      const int fc = t.f0 + (int)rank * feat_per_cta<MODE>();  // this CTA's first feature
      const bool stores = !kChecks || tile_in_range<MODE>(p, t);
      if (!stores && lane == 0) set_error(p.err, ERR_DEVICE_CHECK);
      const int nch = (t.nrows + 31) / 32;
      // Epilogue of chunk ch (32 tokens) from accumulator values v (fp32 bit patterns).
      auto emit = [&](const uint32_t (&v)[32], int ch) {
        if (!stores) return;
        const int nvalid = t.nrows - ch * 32;
        const size_t row0 = (size_t)(t.r0 + ch * 32);
        if (MODE == MODE_UP) {
          // lanes 0..15: gate of features fq + lane; lanes 16..31: up of features fq + lane - 16.
          // Lane l < 16 computes tokens 0..15 with its partner's up values, lane l + 16 tokens
          // 16..31 with its partner's gate values.
          const int fq = fc + q * 16;
          const bool hi = lane >= 16;
          float hv[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const float send = __uint_as_float(hi ? v[i] : v[16 + i]);
            const float recv = __shfl_xor_sync(FULL_MASK, send, 16);
            hv[i] = hi ? silu_mul(recv, __uint_as_float(v[16 + i]))
                       : silu_mul(__uint_as_float(v[i]), recv);
          }
          const int ld = t.shared ? p.S * p.I : p.I;
          store_bf16_chunk<16>(hv, static_cast<__nv_bfloat16*>(t.shared ? p.out1 : p.out0), ld,
                               row0 + (hi ? 16 : 0), nvalid - (hi ? 16 : 0), fq + (lane & 15),
                               fc < feat_total<MODE>(p, t.shared), lane, hint, pol_o);
        } else {
          const int f = fc + q * 32 + lane;                // this thread's feature
          // (feature counts are even, so lanes l and l^1 agree on validity)
          const bool fvalid = f < feat_total<MODE>(p, t.shared);
          if (MODE == MODE_DOWN) {
            float yv[32];
#pragma unroll
            for (int i = 0; i < 32; ++i) yv[i] = __uint_as_float(v[i]);
            store_bf16_chunk<32>(yv, static_cast<__nv_bfloat16*>(t.shared ? p.out1 : p.out0), p.H,
                                 row0, nvalid, f, fvalid, lane, hint, pol_o);
          } else {
            // split-K: partial sums of this split (the reduction adds the bias)
            float* out = (p.splits > 1 ? p.gate_part + (size_t)t.split * p.T * p.N
                                       : static_cast<float*>(p.out0)) + row0 * p.N + f;
            const float bias = (p.splits == 1 && fvalid && p.gate_bias) ? p.gate_bias[f] : 0.0f;
#pragma unroll
            for (int i = 0; i < 32; ++i)
              if (fvalid && i < nvalid) out[(size_t)i * p.N] = __uint_as_float(v[i]) + bias;
          }
        }
      };
      const int pieces = MODE == MODE_GATE ? 0 : (t.split >> 8) & 0xff;
      if (h >= nch) {
        // no chunk of this tile for this warp: the accumulator is free as far as it goes
        __syncwarp();
        if (lane == 0) mbar_arrive_remote(acc ? tempty1 : tempty0);
      } else if (pieces < 2 || !stores) {
        for (int ch = h; ch < nch; ch += 2) {
          uint32_t v[32];
          tmem_ld_32cols(tb + ch * 32, v);
          tmem_wait_ld_fence(v);
          if (ch + 2 >= nch) {
            // this warp's share of the accumulator read: hand it back before the stores
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive_remote(acc ? tempty1 : tempty0);
          }
          emit(v, ch);
        }
      } else {
        // a piece of a split tile: park this warp's share of the partial accumulator (fp32, in
        // L2), count it in; the warp that completes the count adds the pieces in piece order and
        // runs the epilogue for its share, then sets the counter back to zero
        const int piece = t.split & 0xff, sid = t.split >> 16;
        const size_t share = ((size_t)rank * 4 + q) * (TOK * 32);
        float* mine = p.split_part + (size_t)(sid * pieces + piece) * kSplitPieceFloats + share;
        for (int ch = h; ch < nch; ch += 2) {
          uint32_t v[32];
          tmem_ld_32cols(tb + ch * 32, v);
          tmem_wait_ld_fence(v);
          if (ch + 2 >= nch) {
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive_remote(acc ? tempty1 : tempty0);
          }
#pragma unroll
          for (int i = 0; i < 32; ++i)
            if (ch * 32 + i < t.nrows) __stcg(mine + (ch * 32 + i) * 32 + lane, __uint_as_float(v[i]));
        }
        __threadfence();
        __syncwarp();
        int* cnt = p.split_cnt + sid * kSplitWarps + (int)rank * EPI_WARPS + (warp - 2);
        int before = 0;
        if (lane == 0) before = atomicAdd(cnt, 1);
        before = __shfl_sync(FULL_MASK, before, 0);
        if (before == pieces - 1) {
          __threadfence();
          if (lane == 0) atomicExch(cnt, 0);
          const float* all = p.split_part + (size_t)sid * pieces * kSplitPieceFloats + share;
          for (int ch = h; ch < nch; ch += 2) {
            float a[32];
#pragma unroll
            for (int i = 0; i < 32; ++i) a[i] = 0.0f;
            for (int s = 0; s < pieces; ++s) {
              const float* ps = all + (size_t)s * kSplitPieceFloats + (ch * 32) * 32 + lane;
#pragma unroll
              for (int i = 0; i < 32; ++i)
                if (ch * 32 + i < t.nrows) a[i] += __ldcg(ps + i * 32);
            }
            uint32_t v[32];
#pragma unroll
            for (int i = 0; i < 32; ++i) v[i] = __float_as_uint(a[i]);
            emit(v, ch);
          }
        }
      }
      acc ^= 1u;
      if (acc == 0) aphase ^= 1u;
    }
  }

  // both CTAs are done with each other's shared memory, barriers and TMEM before either frees
  tc_fence_before();
  __syncthreads();
  cluster_sync();
  tc_fence_after();
  if (warp == 1) tmem_dealloc_pair(tmem_base, TMEM_COLS);
}

// u[t, e] = gate_bias[e] + sum over splits s (in order) of part[s, t, e]. One thread per output;
// it reads the splits eight at a time, so that a batch of independent loads is in flight before
// the fixed-order sum consumes it.
__global__ void __launch_bounds__(256) gate_reduce_kernel(const float* part, int splits, int T,
                                                          int N, const float* bias, float* u) {
  pdl_wait();
  pdl_trigger();
  const size_t n = (size_t)T * N;
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n;
       i += (size_t)gridDim.x * blockDim.x) {
    float acc = bias ? bias[i % N] : 0.0f;
    for (int s0 = 0; s0 < splits; s0 += 8) {
      float v[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) v[j] = s0 + j < splits ? __ldg(part + (size_t)(s0 + j) * n + i) : 0.0f;
#pragma unroll
      for (int j = 0; j < 8; ++j)
        if (s0 + j < splits) acc += v[j];
    }
    u[i] = acc;
  }
}

// One CTA waits on an mbarrier that nothing ever arrives on; the bounded wait must give up,
// raise the error word and return.
__global__ void wait_selftest_kernel(int* err, unsigned long long timeout_ns) {
  pdl_wait();
  pdl_trigger();
  __shared__ uint64_t b;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&b), 1);
    abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  warp_wait_bounded(smem_u32(&b), 0, &abort_flag, err, timeout_ns);
}

// ---------------------------------------------------------------- host side
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (fn == nullptr) {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  }
  return fn;
}

// 2D bf16 row-major tensor [outer, inner], box [box_outer, 64], 128-byte swizzle.
bool make_map(CUtensorMap* m, const void* base, uint64_t inner, uint64_t outer, uint32_t box_outer) {
  auto fn = encode_fn();
  if (fn == nullptr || base == nullptr || inner == 0 || outer == 0) return false;
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {inner * 2};
  cuuint32_t box[2] = {64, box_outer};
  cuuint32_t es[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box,
            es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// bf16 row-major tensor [outer, inner] (inner a multiple of 64) viewed as (k, row, unit) =
// element (row, 64 unit + k): a box (64, rows, 2) brings `rows` rows of two consecutive 64-element
// units, unit after unit, each a 128-byte-swizzled [rows, 64] tile (the stage layout).
bool make_unit_pair_map(CUtensorMap* m, const void* base, uint64_t inner, uint64_t outer,
                        uint32_t rows) {
  auto fn = encode_fn();
  if (fn == nullptr || base == nullptr || inner == 0 || inner % KU != 0 || outer == 0)
    return false;
  cuuint64_t dims[3] = {(cuuint64_t)KU, outer, inner / KU};
  cuuint64_t strides[2] = {inner * 2, KU * 2};
  cuuint32_t box[3] = {(cuuint32_t)KU, rows, UNITS};
  cuuint32_t es[3] = {1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box,
            es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// UP weights [E, 2I, H] (E experts; rows 0..I-1 gate, I..2I-1 up) as a 5-D tensor
// (k, r, w, g, u) = element (w / 2, (w % 2) * I + 16 g + r, 64 u + k) (w = 2 * expert + gate/up:
// the two halves of an expert and the experts follow each other at the same stride), box
// (64, 16, 2, 4, 2): one load brings 64 features' gate and up rows interleaved 16 at a time
// (gate 16, up 16, ...), for two consecutive 64-element units of the hidden size.
bool make_up_weight_map(CUtensorMap* m, const void* base, uint64_t H, uint64_t I, uint64_t E) {
  auto fn = encode_fn();
  if (fn == nullptr || base == nullptr || H == 0 || H % KU != 0 || I == 0 || I % 64 != 0 ||
      E == 0)
    return false;
  cuuint64_t dims[5] = {(cuuint64_t)KU, 16, 2 * E, I / 16, H / KU};
  cuuint64_t strides[4] = {H * 2, I * H * 2, 16 * H * 2, KU * 2};
  cuuint32_t box[5] = {(cuuint32_t)KU, 16, 2, 4, UNITS};
  cuuint32_t es[5] = {1, 1, 1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 5, const_cast<void*>(base), dims, strides, box,
            es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Token operand [outer, inner]: the unit-pair maps with boxes of 32, 64 and 128 rows.
bool make_token_maps(CUtensorMap (&m)[NTOKMAP], const void* base, uint64_t inner,
                     uint64_t outer) {
  bool ok = true;
  for (int i = 0; i < NTOKMAP; ++i)
    ok = ok && make_unit_pair_map(&m[i], base, inner, outer, 32u << i);
  return ok;
}

// max_pairs > 0 caps the grid at that many CTA pairs.
template <int MODE, int NS>
cudaError_t launch_mode(const TcParams& prm, int num_sms, cudaStream_t st, int max_pairs = 0) {
  static int grid_for_device[64] = {0};
  int dev = 0;
  cudaGetDevice(&dev);
  int grid = (dev >= 0 && dev < 64) ? grid_for_device[dev] : 0;
  cudaLaunchConfig_t cfg;
  memset(&cfg, 0, sizeof(cfg));
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;  // see launch_pdl
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.blockDim = dim3(THREADS, 1, 1);
  cfg.dynamicSmemBytes = smem_bytes();
  cfg.stream = st;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  if (grid == 0) {
    cudaError_t e = cudaFuncSetAttribute(tc_gemm_kernel<MODE, NS>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem_bytes());
    if (e != cudaSuccess) return e;
    // persistent grid: as many CTA pairs as can be resident at once (one CTA per SM)
    cfg.gridDim = dim3(2 * (num_sms / 2), 1, 1);
    int clusters = 0;
    e = cudaOccupancyMaxActiveClusters(&clusters, tc_gemm_kernel<MODE, NS>, &cfg);
    if (e != cudaSuccess) return e;
    if (clusters < 1) return cudaErrorInvalidConfiguration;
    grid = 2 * (clusters < num_sms / 2 ? clusters : num_sms / 2);
    if (dev >= 0 && dev < 64) grid_for_device[dev] = grid;
  }
  if (max_pairs > 0 && 2 * max_pairs < grid) grid = 2 * max_pairs;
  cfg.gridDim = dim3(grid, 1, 1);
  note_launches(1);
  return cudaLaunchKernelEx(&cfg, tc_gemm_kernel<MODE, NS>, prm);
}

}  // namespace

cudaError_t launch_gemm_tc(const GemmArgs& a, int num_sms, cudaStream_t st) {
  if (a.T <= 0) return cudaSuccess;
  TcParams prm;
  memset(&prm, 0, sizeof(prm));
  prm.offsets = a.offsets;
  prm.rows_cap = a.rows_cap;
  prm.n_routed = a.n_routed;
  prm.has_shared = a.has_shared;
  prm.T = a.T; prm.H = a.H; prm.I = a.I; prm.S = a.S; prm.N = a.N;
  prm.out0 = a.out0; prm.out1 = a.out1;
  prm.gate_bias = a.gate_bias;
  prm.splits = 1;
  prm.err = a.err;
  prm.sched = a.mode == MODE_GATE ? nullptr : a.sched;
  // small batches: every weight tile is read by one CTA pair, while the token rows and outputs are
  // read again by the next stage (x_perm / h / y_perm fit in L2)
  prm.l2_hints = (a.mode != MODE_GATE && a.T <= kL2HintMaxTokens) ? 1 : 0;
  prm.offsets_early = a.mode != MODE_GATE ? a.offsets_early : 0;
  if (a.mode != MODE_GATE && a.sched != nullptr) {
    prm.split_part = a.split_part;
    prm.split_cnt = a.split_cnt;
  }
  const uint64_t H = a.H, I = a.I, S = a.S, N = a.N, T = a.T, R = a.rows_cap;
  bool ok = true;
  if (a.mode == MODE_GATE) {
    ok = make_unit_pair_map(&prm.tmW0, a.b0, H, N, BM) && make_token_maps(prm.tmX0, a.a0, H, T);
    if (!ok) return cudaErrorInvalidValue;
    // Few token tiles (decode): split the K range over up to kGateMaxSplits pairs per tile; the
    // partial sums go to the caller's scratch and are reduced in a fixed order. (Measured at
    // 32-512 tokens: more, shorter splits only add partial traffic; 16 is 1-3 us faster than
    // one split per pair.)
    const int tiles = (int)((T + TOK - 1) / TOK) * (int)((N + 2 * BM - 1) / (2 * BM));
    const int ku_total = (int)(H / KU);
    const int kb_total = (ku_total + UNITS - 1) / UNITS;
    const int pairs = num_sms / 2;
    if (a.gate_part != nullptr && 2 * tiles <= pairs) {
      int want = min(pairs / tiles, kGateMaxSplits);
      const size_t fit = a.gate_part_floats / ((size_t)T * N);
      if ((size_t)want > fit) want = (int)fit;
      if (want > kb_total) want = kb_total;
      if (want > 1) {
        const int kb_per_split = (kb_total + want - 1) / want;
        prm.ku_per_split = kb_per_split * UNITS;
        prm.splits = (kb_total + kb_per_split - 1) / kb_per_split;
        prm.gate_part = a.gate_part;
      }
    }
    // one pair per work item (the items are fewer than the pairs whenever K is split)
    const int items = tiles * prm.splits;
    cudaError_t e = launch_mode<MODE_GATE, 3>(prm, num_sms, st, items < pairs ? items : 0);
    if (e != cudaSuccess || prm.splits == 1) return e;
    int blocks = (int)(((size_t)T * N + 255) / 256);
    if (blocks > num_sms * 8) blocks = num_sms * 8;
    return launch_pdl(gate_reduce_kernel, dim3(blocks), dim3(256), 0, st,
                      static_cast<const float*>(a.gate_part), prm.splits, (int)T, (int)N,
                      a.gate_bias, static_cast<float*>(a.out0));
  }
  if (a.mode == MODE_UP) {
    if (a.n_routed > 0) {
      ok = ok && make_up_weight_map(&prm.tmW0, a.b0, H, I, N);
      if (a.row_token != nullptr) {
        ok = ok && make_map(&prm.tmXg, a.a0, H, T, 1);  // x [T, H], rows gathered
        prm.row_token = a.row_token;
      } else {
        ok = ok && make_token_maps(prm.tmX0, a.a0, H, R);
      }
    }
    if (a.has_shared) ok = ok && make_up_weight_map(&prm.tmW1, a.b1, H, I, S) &&
                           make_token_maps(prm.tmX1, a.a1, H, T);
    if (!ok) return cudaErrorInvalidValue;
    return prm.T <= kDeepRingMaxTokens ? launch_mode<MODE_UP, NSLOT>(prm, num_sms, st)
                                       : launch_mode<MODE_UP, 3>(prm, num_sms, st);
  }
  if (a.n_routed > 0) ok = ok && make_unit_pair_map(&prm.tmW0, a.b0, I, N * H, BM) &&
                           make_token_maps(prm.tmX0, a.a0, I, R);
  if (a.has_shared) ok = ok && make_unit_pair_map(&prm.tmW1, a.b1, I, S * H, BM) &&
                         make_token_maps(prm.tmX1, a.a1, S * I, T);
  if (!ok) return cudaErrorInvalidValue;
  return prm.T <= kDeepRingMaxTokens ? launch_mode<MODE_DOWN, NSLOT>(prm, num_sms, st)
                                     : launch_mode<MODE_DOWN, 3>(prm, num_sms, st);
}

cudaError_t launch_wait_selftest(int* err, unsigned long long timeout_ns, cudaStream_t st) {
  return launch_pdl(wait_selftest_kernel, dim3(1), dim3(32), 0, st, err, timeout_ns);
}

}  // namespace moe

