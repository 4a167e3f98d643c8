// Dense GEMM on the 5th-generation tensor cores (tcgen05) of sm_103a: FP16
// (or BF16) operands on kind::f16, and block-scaled 4-bit operands (MXFP4:
// E2M1 codes with an E8M0 scale per 32 values along K) on kind::mxf4.
//
//   D[M x N] = epilogue(alpha * A[M x K] . B[N x K]^T + beta * C)
//
// The contraction the "DeepGEMM" articles build their tile planner around
// (discosf.com/news/5532976, section 3.2: a 4096^3 FP16 GEMM; section 3.5:
// FP32 accumulation, FP16 output; kwkr.cn/news/562171, section 2.2 first and
// third layers: planned tiles and a fused epilogue).  The pages target
// warp-level mma.sync on A100/H100; on Blackwell the same contraction maps to
// a single-thread-issued tcgen05.mma with the accumulator in tensor memory:
//
//   warp 0      TMA producer: a ring of `Stages` shared-memory slots, each a
//               128 x 64 tile of A and a B tile (128-byte swizzle);
//   warp 1      MMA issuer: 4 x tcgen05.mma (K = 16 each) per slot into an
//               FP32 accumulator in TMEM; tcgen05.commit frees slots;
//   warp 2      allocates / frees the tensor memory (2 accumulators);
//   warps 4-11  epilogue: tcgen05.ld of the accumulator (warps w and w + 4
//               own TMEM lanes 32*(w % 4) .. +31 = rows, and half of the
//               columns each), alpha/beta/bias/GELU in FP32, FP16
//               round-to-nearest-even.  With N % 8 == 0 each warp moves C in
//               and D out as 32 x 32 boxes through two shared-memory staging
//               buffers with TMA (whole lines, C loaded ahead of use); other
//               shapes store from registers.
//
// CG = 1: one CTA computes a 128 x BN tile.
// CG = 2: a cluster of two CTAs computes a 256 x BN tile with 256-row MMAs
//   (cta_group::2).  Each CTA loads its own 128 rows of A and BN/2 rows of B;
//   the even CTA issues the MMAs, which read both CTAs' shared memory, and its
//   commits arrive on the barriers of both CTAs.  Every A and B tile is read
//   from L2 once per pair instead of once per CTA, halving L2->SM traffic per
//   FLOP, and each SM's shared memory feeds half of the B operand.
//
// MXFP4: a stage holds 128 bytes of packed codes per row (256 values of K,
// as 16-bit stages hold 64), loaded by TMA as bytes into the same swizzled
// slots, plus the stage's E8M0 scales: TMA brings 16 row-major scale bytes
// per row of A and B (the stage's 8 and the next stage's), warp 3 rearranges
// the stage's into the interleaved images the MMA thread copies into tensor
// memory (tcgen05.cp, in issue order with its MMAs), and the MMA thread
// issues four block-scaled MMAs of K = 64 per stage: the 4-bit codes reach
// the tensor cores as they are stored, with no 16-bit copy (discosf.com/news/5532976, section 4.3: packed 4-bit weights instead
// of an FP16 emulation; section 2.2, layer 2: each precision in the tensor
// core's own format).
//
// The kernel is persistent (one CTA / pair per SM / SM pair walks the tile
// list), and the two TMEM accumulators let the epilogue of tile i overlap the
// main loop of tile i+1.  Out-of-range rows and K columns are zero-filled by
// TMA; the epilogue masks (or the store's tensor map clips) rows >= M and
// columns >= N.  Operand tiles are loaded with an L2 evict-last hint (they
// are re-read by other tiles), C with evict-first.  Launches use programmatic
// dependent launch: set-up overlaps the previous kernel's drain, and global
// memory is touched only after griddepcontrol.wait.  Every mbarrier wait is
// bounded: on a timeout the CTA records it in the status word, drains its
// own copies and MMAs, frees its tensor memory and exits.
#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <algorithm>

#include "tc_common.cuh"

namespace dg {
namespace {

using tc::kBlockK;
using tc::kBlockM;
constexpr int kThreads = 384;
constexpr int kEpiWarp0 = 4;
constexpr int kEpiWarps = 8;  // two warps per 32-lane TMEM quarter, each half of the columns
constexpr int kTileBytesA = kBlockM * kBlockK * 2;

struct TcParams {
  int M, N, K;
  int num_m_blocks, num_n_blocks, num_tiles, num_k_blocks;
  int group_m;
  Epi epi;
  const void* C;  // read when beta != 0 (FP16, or INT32 when Out == kOutI32)
  int64_t ldc;
  void* D;
  int64_t ldd;
  const __half* bias;
  int32_t alpha_i, beta_i;  // integer scalars of the INT32 output
  int* status;
  uint64_t timeout_ns;
  uint32_t stage_tx;  // bytes TMA delivers per stage (both CTAs of a pair)
  int staged;         // FP16 out through shared-memory boxes and TMA (else direct stores)
  uint32_t idesc_ab;  // instruction-descriptor bits of the operand type (0: FP16; BF16 bits)
};
static_assert(sizeof(TcParams) <= 128, "parameter struct within 128 bytes (see Epi)");

// Stream-K division of the work (kwkr.cn/news/562171, section 2.2 first
// layer: a K step chosen per piece of work, so that ragged tile counts
// still fill every SM).  Tiles [0, dp_tiles) are whole work units, walked as
// in the data-parallel kernel (unit u takes u, u + units, ...).  The K
// blocks of tiles [dp_tiles, num_tiles), taken tile after tile, form one
// sequence of sk_iters iterations that is cut into sk_units contiguous
// ranges of equal length (+-1), unit u < sk_units taking range u after its
// whole tiles.  A tile that several ranges meet is finished by the unit
// holding its first K block (piece 0), which meets it last in its range;
// every later piece q stores its FP32 partial accumulator in slot q - 1 of
// the tile and raises one flag per epilogue warp, and piece 0 adds the
// partials to its own in piece order (a fixed order: the result does not
// depend on timing).  Flags hold the launch's epoch + 1, read from sync[0]
// at the start; the last CTA to finish advances the epoch (sync[1] counts
// finished CTAs), so flags left by an earlier or an aborted launch never
// match.
struct SkParams {
  int dp_tiles;      // tiles walked whole (num_tiles without stream-K)
  int sk_units;      // units holding a range (0: none)
  int64_t sk_iters;  // (num_tiles - dp_tiles) * num_k_blocks
  int max_pieces;    // most ranges a tile meets; partial slots per tile: max_pieces - 1
  float* partial;    // [tile - dp_tiles][piece - 1][kBlockM * CG][BN]
  unsigned* sync;    // [0] epoch, [1] CTAs finished, then flags
                     // [tile - dp_tiles][piece - 1][CG][kEpiWarps]
};

// One unit's piece of work: K blocks [kb0, kb1) of tile t.  pieces == 1: the
// whole tile; else piece 0 finishes the tile and pieces > 0 store partials.
struct Work {
  int t, kb0, kb1, piece, pieces;
};

// A unit's position in its list of works: the next whole tile, then the
// stream-K iterations [it, it_end) still to take.
struct WorkWalk {
  int t;
  int64_t it, it_end;
};

__device__ __forceinline__ int64_t sk_range_begin(const SkParams& s, int u) {
  return static_cast<int64_t>(u) * s.sk_iters / s.sk_units;
}

// The unit whose range holds stream-K iteration i: the largest u with
// sk_range_begin(u) <= i.
__device__ __forceinline__ int sk_unit_of(const SkParams& s, int64_t i) {
  return static_cast<int>(((i + 1) * s.sk_units - 1) / s.sk_iters);
}

template <bool SK>
__device__ __forceinline__ WorkWalk walk_start(const SkParams& s, int unit0) {
  WorkWalk w{unit0, 0, 0};
  if (SK && unit0 < s.sk_units) {
    w.it = sk_range_begin(s, unit0);
    w.it_end = sk_range_begin(s, unit0 + 1);
  }
  return w;
}

// The unit's next work, false past its last.
template <bool SK>
__device__ __forceinline__ bool walk_next(WorkWalk& w, const TcParams& p, const SkParams& s,
                                          int unit0, int units, Work& out) {
  const int dp_end = SK ? s.dp_tiles : p.num_tiles;
  if (w.t < dp_end) {
    out = Work{w.t, 0, p.num_k_blocks, 0, 1};
    w.t += units;
    return true;
  }
  if (!SK || w.it >= w.it_end) return false;
  const int kbn = p.num_k_blocks;
  const int64_t ts = w.it / kbn;
  const int kb0 = static_cast<int>(w.it - ts * kbn);
  const int64_t left = w.it_end - w.it;
  const int kb1 = left < kbn - kb0 ? kb0 + static_cast<int>(left) : kbn;
  const int first = sk_unit_of(s, ts * kbn);
  const int last = sk_unit_of(s, ts * kbn + kbn - 1);
  out = Work{s.dp_tiles + static_cast<int>(ts), kb0, kb1, unit0 - first, last - first + 1};
  w.it += kb1 - kb0;
  return true;
}

// A work whose accumulator goes to a partial slot instead of D.
__device__ __forceinline__ bool sk_writer(const Work& w) { return w.pieces > 1 && w.piece > 0; }

// The tile of the unit's idx-th work that writes D (-1: none).
template <bool SK>
__device__ __forceinline__ int nth_output_tile(const TcParams& p, const SkParams& s, int unit0,
                                               int units, int idx) {
  if (!SK) {
    const int t = unit0 + idx * units;
    return t < p.num_tiles ? t : -1;
  }
  WorkWalk w = walk_start<SK>(s, unit0);
  Work wk;
  while (walk_next<SK>(w, p, s, unit0, units, wk))
    if (!sk_writer(wk) && idx-- == 0) return wk.t;
  return -1;
}

// Output modes: FP16 with the fused epilogue, or exact INT32 for INT8 inputs
// widened to FP16 (K accumulated in exact FP32 chunks, INT32 running sum).
enum : int { kOutF16 = 0, kOutI32 = 1 };

// Operand kinds: 16-bit (FP16, or BF16 with the BF16 operand bits), or
// packed E2M1 with E8M0 block scales (MXFP4) on the block-scaled MMA.  An
// MXFP4 stage holds the same 128 bytes per row as a 16-bit stage (256 codes
// instead of 64 values), so the ring, the TMA boxes and the shared-memory
// descriptors are the same; each stage adds the scales of its 256-wide K
// block: 8 bytes per row, as two 512-byte images of 32 lines x 16 bytes for
// each 128 rows (line r, word i, byte k: the scale of row 32 i + r for the
// K block's 32-value block 4 j + k, image j).
enum : int { kKind16 = 0, kKindMx = 1 };
constexpr int kMxSfImage = 512;           // one image: 128 rows x 4 scales
constexpr int kMxSfRowBlock = 2 * kMxSfImage;  // 128 rows x the 8 scales of a stage

// Shared memory: the operand ring, then two staging boxes per epilogue warp,
// then the barriers.
template <int BN, int Stages, int CG, int Kind = kKind16>
struct TcSmem {
  static constexpr int kRowsB = BN / CG;  // B rows this CTA loads
  static constexpr int kTileBytesB = kRowsB * kBlockK * 2;
  // MXFP4, per stage: the scale images, this CTA's 128 rows of A, then the
  // whole B tile's rows in 128-row blocks (a CTA pair's MMA reads every
  // column's scales in each CTA's tensor memory); and the row-major scale
  // bytes they are built from, 16 per row (this CTA's 128 rows of A, then
  // the B tile's BN rows)
  static constexpr int kSfBlocksB = (BN + 127) / 128;
  static constexpr int kSfBytes = Kind == kKindMx ? kMxSfRowBlock * (1 + kSfBlocksB) : 0;
  static constexpr int kSfRowsBytes = Kind == kKindMx ? 16 * (kBlockM + BN) : 0;
  static constexpr int kOffA = 0;
  static constexpr int kOffB = kOffA + Stages * kTileBytesA;
  static constexpr int kOffSf = kOffB + Stages * kTileBytesB;
  static constexpr int kOffSfRows = kOffSf + Stages * kSfBytes;
  static constexpr int kOffEpi = kOffSfRows + Stages * kSfRowsBytes;
  static constexpr int kEpiBytes = kEpiWarps * 2 * tc::kEpiBoxBytes;
  static constexpr int kOffBar = kOffEpi + kEpiBytes;
  // full[Stages], empty[Stages], tmem_full[2], tmem_empty[2], drain, one
  // C-load barrier per staging box, then (MXFP4) sf_full[Stages] (the
  // stage's scale bytes landed) and img_ready[Stages] (its images built)
  static constexpr int kNumBars = 2 * Stages + 5 + 2 * kEpiWarps + (Kind == kKindMx ? 2 * Stages : 0);
  static constexpr int kOffTmemSlot = kOffBar + kNumBars * 8;
  static constexpr int kOffAbort = kOffTmemSlot + 4;
  static constexpr int kBytes = kOffAbort + 4;
  static constexpr int kLaunchBytes = kBytes + 1024;  // room to align the base to 1 KB
  static_assert(kLaunchBytes <= 232448, "shared memory of one CTA");
  static_assert(kTileBytesB % 1024 == 0, "B tiles keep 1 KB alignment");
  static_assert(kOffSfRows % 128 == 0 && kSfRowsBytes % 128 == 0, "TMA destinations aligned");
};

__device__ __forceinline__ bool aborted(volatile int* flag) { return *flag != 0; }

// MXFP4 scale images.  A pair of K blocks (2 kp, 2 kp + 1) has its scale
// bytes loaded once, 16 per row (this CTA's 128 rows of A, then the B
// tile's BN rows): bytes 0..7 are K block 2 kp's 8 scales, 8..15 the next
// one's.  Lane r of the building warp reads rows r, 32 + r, 64 + r and
// 96 + r of each 128-row block (whole 16-byte rows: a warp's reads are free
// of bank conflicts); B rows past BN read 0.
template <int BN>
struct MxScaleRows {
  static constexpr int kBlocks = 1 + (BN + 127) / 128;  // A, then B's 128-row blocks
  uint4 v[kBlocks][4];
  __device__ __forceinline__ void load(const uint8_t* rows, int r) {
#pragma unroll
    for (int blk = 0; blk < kBlocks; ++blk)
#pragma unroll
      for (int w = 0; w < 4; ++w) {
        const int row = (blk == 0 ? 0 : kBlockM + 128 * (blk - 1)) + 32 * w + r;
        v[blk][w] = (blk == 0 || row - kBlockM < BN)
                        ? *reinterpret_cast<const uint4*>(rows + 16 * row)
                        : make_uint4(0u, 0u, 0u, 0u);
      }
  }
  // Line r of both images of every block for the pair's first (second) K
  // block: image j line r = the 4 scales 4 j .. 4 j + 3 of the four rows.
  __device__ __forceinline__ void store(uint8_t* img, int r, bool second) const {
#pragma unroll
    for (int blk = 0; blk < kBlocks; ++blk) {
      uint8_t* dst = img + blk * kMxSfRowBlock + r * 16;
      const uint4* q = v[blk];
      if (second) {
        *reinterpret_cast<uint4*>(dst) = make_uint4(q[0].z, q[1].z, q[2].z, q[3].z);
        *reinterpret_cast<uint4*>(dst + kMxSfImage) = make_uint4(q[0].w, q[1].w, q[2].w, q[3].w);
      } else {
        *reinterpret_cast<uint4*>(dst) = make_uint4(q[0].x, q[1].x, q[2].x, q[3].x);
        *reinterpret_cast<uint4*>(dst + kMxSfImage) = make_uint4(q[0].y, q[1].y, q[2].y, q[3].y);
      }
    }
  }
};

// Staged epilogue: epilogue warp wi (0..7) owns TMEM lane quarter wi & 3 and
// half wi >> 2 of the tile's 32-column chunks.  Its chunks form one stream over
// the tiles the CTA writes to D.  Returns the D coordinates of chunk k of the
// warp's share of tile t, false when the box lies wholly outside D.
template <int BN, int CG>
__device__ __forceinline__ bool epi_box(const TcParams& p, int t, uint32_t rank, int wi, int k,
                                        int& x, int& y) {
  constexpr int kChunks = BN / 32;
  const int lo = (wi >> 2) == 0 ? 0 : (kChunks + 1) / 2;
  int mb, nb;
  tc::tile_coords(t, p.num_m_blocks, p.num_n_blocks, p.group_m, mb, nb);
  x = nb * BN + (lo + k) * 32;
  y = mb * kBlockM * CG + static_cast<int>(rank) * kBlockM + (wi & 3) * 32;
  return x < p.N && y < p.M;
}

// Loads C of chunk k of warp wi's share of tile t (stream chunk j) into its
// box j & 1 (arriving on that box's barrier).  For the first chunk of a tile
// it also asks L2 for the share's chunks from the third on, which are loaded
// only during the epilogue.  Box j & 1 must no longer feed a store.
template <int BN, int CG>
__device__ __forceinline__ void epi_load_c(const CUtensorMap* map, const TcParams& p, int t,
                                           uint32_t rank, int wi, int k, int j, uint8_t* boxes,
                                           uint64_t* cbar, uint64_t policy) {
  constexpr int kChunks = BN / 32;
  const int n = (wi >> 2) == 0 ? (kChunks + 1) / 2 : kChunks - (kChunks + 1) / 2;
  int x, y;
  if (t < 0 || !epi_box<BN, CG>(p, t, rank, wi, k, x, y)) return;
  const int b = j & 1;
  mbar_arrive_expect_tx(&cbar[b], tc::kEpiBoxBytes);
  tma_load_2d(map, &cbar[b], boxes + b * tc::kEpiBoxBytes, x, y, policy);
  if (k == 0)
    for (int kk = 2; kk < n; ++kk)
      if (epi_box<BN, CG>(p, t, rank, wi, kk, x, y)) tma_prefetch_l2_2d(map, x, y);
}

template <int BN, int Stages, int CG, int Out, int Kind, bool SK>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_tc_kernel(const __grid_constant__ CUtensorMap tmap_a,
                       const __grid_constant__ CUtensorMap tmap_b,
                       const __grid_constant__ CUtensorMap tmap_c,
                       const __grid_constant__ CUtensorMap tmap_d,
                       const __grid_constant__ CUtensorMap tmap_sfa,
                       const __grid_constant__ CUtensorMap tmap_sfb, const TcParams p,
                       const __grid_constant__ EpiProgram prog, const SkParams sk) {
  using L = TcSmem<BN, Stages, CG, Kind>;
  constexpr bool kMx = Kind == kKindMx;
  static_assert(!kMx || Out == kOutF16, "MXFP4: FP16 output");
  // Stream-K: 16-bit operands, FP16 output through the staged epilogue, and
  // at least two 32-column chunks per epilogue warp (so that the producer's
  // first two C boxes belong to one tile)
  static_assert(!SK || (Kind == kKind16 && Out == kOutF16 && BN >= 128), "stream-K variant");
  // two FP32 accumulators (the INT32 mode keeps its running sums in registers);
  // MXFP4 adds two buffers of scale words after them: A's 128 rows (4
  // columns per scale word, one per 32-row group) and B's rows (one column
  // per 32 rows) for the two words of a stage
  constexpr int kSfColsA = 8;
  constexpr int kSfColsB = 8 * L::kSfBlocksB;
  constexpr int kSfCols = kSfColsA + kSfColsB;
  constexpr int kColsNeeded = 2 * BN + (kMx ? 2 * kSfCols : 0);
  constexpr int kTmemCols = kColsNeeded <= 128 ? 128 : (kColsNeeded <= 256 ? 256 : 512);
  static_assert(kColsNeeded <= 512, "tensor memory");
  // K blocks per accumulation chunk: the whole K, or exact-FP32 chunks
  const int chunk_kb = Out == kOutI32 ? tc::kI32ChunkKb : p.num_k_blocks;
  const int num_chunks = (p.num_k_blocks + chunk_kb - 1) / chunk_kb;
  constexpr int kTileM = kBlockM * CG;  // rows of D per tile
  const uint32_t idesc = idesc_f16_f32(kTileM, BN) | p.idesc_ab;

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t* smem_a = smem + L::kOffA;
  uint8_t* smem_b = smem + L::kOffB;
  uint8_t* smem_sf = smem + L::kOffSf;
  uint8_t* smem_sf_rows = smem + L::kOffSfRows;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::kOffBar);
  uint64_t* full_bar = bars;
  uint64_t* empty_bar = bars + Stages;
  uint64_t* tmem_full = bars + 2 * Stages;
  uint64_t* tmem_empty = bars + 2 * Stages + 2;
  uint64_t* drain_bar = bars + 2 * Stages + 4;
  uint64_t* epi_bar = bars + 2 * Stages + 5;  // [kEpiWarps][2]
  uint64_t* sf_full = epi_bar + 2 * kEpiWarps;  // MXFP4 only
  uint64_t* img_ready = sf_full + Stages;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::kOffTmemSlot);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::kOffAbort);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = CG == 2 ? cluster_ctarank() : 0u;
  const bool leader = rank == 0;
  const int unit0 = CG == 2 ? static_cast<int>(blockIdx.x >> 1) : static_cast<int>(blockIdx.x);
  const int units = CG == 2 ? static_cast<int>(gridDim.x >> 1) : static_cast<int>(gridDim.x);

  if (threadIdx.x == 0) {
    for (int s = 0; s < Stages; ++s) {
      mbar_init(&full_bar[s], 1);
      mbar_init(&empty_bar[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&tmem_full[b], 1);
      mbar_init(&tmem_empty[b], CG * kEpiWarps * 32);  // every epilogue thread of the pair
    }
    mbar_init(drain_bar, 1);
    for (int b = 0; b < 2 * kEpiWarps; ++b) mbar_init(&epi_bar[b], 1);
    if (kMx) {
      for (int s = 0; s < Stages; ++s) {
        mbar_init(&sf_full[s], 1);
        mbar_init(&img_ready[s], CG);  // the building warp of each CTA of the pair
      }
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmap_a);
    tma_prefetch_desc(&tmap_b);
    if (kMx) {
      tma_prefetch_desc(&tmap_sfa);
      tma_prefetch_desc(&tmap_sfb);
    }
    if (p.staged) {
      tma_prefetch_desc(&tmap_d);
      if (Out == kOutF16 && p.epi.beta != 0.0f) tma_prefetch_desc(&tmap_c);
    }
  }
  if (warp == 2) {
    if (CG == 2)
      tmem_alloc_pair<kTmemCols>(tmem_slot);
    else
      tmem_alloc<kTmemCols>(tmem_slot);
  }
  tc_fence_before_sync();
  __syncthreads();
  if (CG == 2) cluster_sync();  // peer barriers initialised before any remote arrive
  tc_fence_after_sync();
  const uint32_t tmem_base = *tmem_slot;
  bool ok = true;
  // Launched with programmatic stream serialization: the kernel before this
  // one in the stream may still be finishing.  Everything above touched only
  // this CTA's (or pair's) own on-chip state; global memory waits for it.
  grid_dependency_wait();

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (elect_one_lane()) {
      // Operand tiles are read again by other tiles: they outrank C and D in L2.
      const uint64_t pol = policy_evict_last();
      // The staged epilogue's first two C boxes per warp are loaded from here,
      // behind the first ring of operand tiles, so they do not delay the first MMA.
      const bool first_c = Out == kOutF16 && p.staged && p.epi.beta != 0.0f;
      auto initial_c = [&]() {
        const uint64_t pol_c = policy_evict_first();
        constexpr int kChunks = BN / 32;
        const int t0 = nth_output_tile<SK>(p, sk, unit0, units, 0);
        const int t1 = nth_output_tile<SK>(p, sk, unit0, units, 1);
        for (int wi = 0; wi < kEpiWarps; ++wi) {
          const int n = (wi >> 2) == 0 ? (kChunks + 1) / 2 : kChunks - (kChunks + 1) / 2;
          for (int j = 0; j < 2; ++j)
            epi_load_c<BN, CG>(&tmap_c, p, j < n ? t0 : t1, rank, wi, j % n, j,
                               smem + L::kOffEpi + wi * 2 * tc::kEpiBoxBytes, epi_bar + wi * 2,
                               pol_c);
        }
      };
      int stage = 0;
      uint32_t phase = 0;
      int64_t issued = 0;
      // MXFP4: ring slots whose latest fill loaded scale bytes, and per slot
      // the parity of the scale loads so far (a slot that holds an odd K
      // block loads none, so these phases do not follow the ring's)
      uint32_t sf_slots = 0, sf_loads = 0;
      // The data-parallel kernel walks its tiles in a plain loop with constant
      // K bounds: taking them from the work in registers slowed the
      // single-thread issue loops measurably (FP16 2048^3 +6%, MXFP4 4096^3 +5%).
      WorkWalk walk = walk_start<SK>(sk, unit0);
      Work wk;
      for (int t = unit0;
           SK ? (ok && walk_next<SK>(walk, p, sk, unit0, units, wk)) : (t < p.num_tiles && ok);
           t += units) {
        if constexpr (!SK) wk = Work{t, 0, p.num_k_blocks, 0, 1};
        int m_blk, n_blk;
        tc::tile_coords(wk.t, p.num_m_blocks, p.num_n_blocks, p.group_m, m_blk, n_blk);
        const int a_row = m_blk * kTileM + static_cast<int>(rank) * kBlockM;
        const int b_row = n_blk * BN + static_cast<int>(rank) * L::kRowsB;
        for (int kb = SK ? wk.kb0 : 0; kb < (SK ? wk.kb1 : p.num_k_blocks); ++kb) {
          if (!mbar_wait_abortable(&empty_bar[stage], phase ^ 1, p.timeout_ns, p.status,
                                   abort_flag)) {
            ok = false;
            break;
          }
          if (kMx && (kb & 1) == 0) {
            // The scale bytes of K blocks kb and kb + 1, on this CTA's own
            // barrier, ahead of the operand tiles so that the images are
            // built while those land: 16 per row (x = 8 kb, on a 16-byte
            // boundary as TMA needs), this CTA's rows of A and the whole B
            // tile's rows.
            uint8_t* dst_rows = smem_sf_rows + stage * L::kSfRowsBytes;
            mbar_arrive_expect_tx(&sf_full[stage], L::kSfRowsBytes);
            tma_load_2d(&tmap_sfa, &sf_full[stage], dst_rows, 8 * kb, a_row, pol);
            tma_load_2d(&tmap_sfb, &sf_full[stage], dst_rows + 16 * kBlockM, 8 * kb, n_blk * BN,
                        pol);
            sf_slots |= 1u << stage;
            sf_loads ^= 1u << stage;
          } else if (kMx) {
            sf_slots &= ~(1u << stage);
          }
          uint8_t* dst_a = smem_a + stage * kTileBytesA;
          uint8_t* dst_b = smem_b + stage * L::kTileBytesB;
          if (CG == 1) {
            mbar_arrive_expect_tx(&full_bar[stage], p.stage_tx);
            // x counts elements of the map: FP16 values, or bytes of two codes
            tma_load_2d(&tmap_a, &full_bar[stage], dst_a, kb * (kMx ? 128 : kBlockK), a_row, pol);
            tma_load_2d(&tmap_b, &full_bar[stage], dst_b, kb * (kMx ? 128 : kBlockK), b_row, pol);
          } else {
            // both CTAs' copies complete on the even CTA's full barrier
            if (leader) mbar_arrive_expect_tx(&full_bar[stage], p.stage_tx);
            const uint32_t bar0 = mapa_shared(smem_addr(&full_bar[stage]), 0);
            tma_load_2d_pair(&tmap_a, bar0, dst_a, kb * (kMx ? 128 : kBlockK), a_row, pol);
            tma_load_2d_pair(&tmap_b, bar0, dst_b, kb * (kMx ? 128 : kBlockK), b_row, pol);
          }
          ++issued;
          if (first_c && issued == Stages) initial_c();
          if (++stage == Stages) {
            stage = 0;
            phase ^= 1;
          }
        }
      }
      if (first_c && ok && issued < Stages) initial_c();
      // Every operand load is issued: a kernel launched after this one may be
      // scheduled now (not earlier: small blocks of another kernel that fit
      // beside this CTA would wait on its SM for the whole main loop).
      grid_launch_dependents();
      if (!ok) {
        *abort_flag = 1;
        // Let the copies this thread started land before the CTA goes away.
        const int64_t first = issued > Stages ? issued - Stages : 0;
        for (int64_t i = first; i < issued; ++i) {
          const uint32_t par = static_cast<uint32_t>((i / Stages) & 1);
          if (CG == 1 || leader) mbar_wait(&full_bar[i % Stages], par, p.timeout_ns, p.status);
          // a slot's latest scale load completes the phase of parity loads - 1
          if (kMx && ((sf_slots >> (i % Stages)) & 1u))
            mbar_wait(&sf_full[i % Stages], ((sf_loads >> (i % Stages)) & 1u) ^ 1u, p.timeout_ns,
                      p.status);
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (leader && elect_one_lane()) {
      int stage = 0;
      uint32_t phase = 0;
      int acc = 0;
      uint32_t acc_phase = 0;
      int sf_buf = 0;  // MXFP4: scale buffer of the next stage
      WorkWalk walk = walk_start<SK>(sk, unit0);
      Work wk;
      for (int t = unit0;
           SK ? (ok && walk_next<SK>(walk, p, sk, unit0, units, wk)) : (t < p.num_tiles && ok);
           t += units) {
        if constexpr (!SK) wk = Work{t, 0, p.num_k_blocks, 0, 1};
        for (int ch = 0; ch < num_chunks && ok; ++ch) {
          if (!mbar_wait_abortable(&tmem_empty[acc], acc_phase ^ 1, p.timeout_ns, p.status,
                                   abort_flag)) {
            ok = false;
            break;
          }
          tc_fence_after_sync();
          const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * BN);
          const int kb0 = SK ? wk.kb0 + ch * chunk_kb : ch * chunk_kb;
          const int kb1 = SK ? min(wk.kb1, kb0 + chunk_kb) : min(p.num_k_blocks, kb0 + chunk_kb);
          for (int kb = kb0; kb < kb1; ++kb) {
            if (!mbar_wait_abortable(&full_bar[stage], phase, p.timeout_ns, p.status,
                                     abort_flag) ||
                (kMx && !mbar_wait_abortable(&img_ready[stage], phase, p.timeout_ns, p.status,
                                             abort_flag))) {
              ok = false;
              break;
            }
            tc_fence_after_sync();
            // K step k of the stage starts 32 bytes further into the swizzled
            // rows: +2 in the descriptor's 16-byte address field
            const uint64_t da0 = smem_desc_sw128(smem_addr(smem_a + stage * kTileBytesA));
            const uint64_t db0 = smem_desc_sw128(smem_addr(smem_b + stage * L::kTileBytesB));
            if (kMx) {
              // The stage's scale images into scale buffer sf_buf: A's two
              // words (4 columns each), then B's (one column per 32 rows of
              // each 128-row block, 8 columns per block and word).  The copies
              // run before this thread's later MMAs, in issue order; the MMAs
              // of the stage before read the other buffer.
              const uint32_t sfa_t = tmem_base + static_cast<uint32_t>(2 * BN + sf_buf * kSfCols);
              const uint32_t sfb_t = sfa_t + kSfColsA;
              const uint32_t src = smem_addr(smem_sf + stage * L::kSfBytes);
#pragma unroll
              for (int w = 0; w < 2; ++w) {
                // a pair's copy fills both CTAs' tensor memory, each from its
                // own shared memory at the same offset
                const uint32_t sa = sfa_t + 4 * w;
                const uint64_t da = smem_desc_rows16(src + w * kMxSfImage);
                if (CG == 2)
                  tc_cp_32x128b_warpx4_pair(sa, da);
                else
                  tc_cp_32x128b_warpx4(sa, da);
#pragma unroll
                for (int h = 0; h < L::kSfBlocksB; ++h) {
                  const uint32_t sb = sfb_t + w * 4 * L::kSfBlocksB + 4 * h;
                  const uint64_t db = smem_desc_rows16(src + kMxSfRowBlock * (1 + h) + w * kMxSfImage);
                  if (CG == 2)
                    tc_cp_32x128b_warpx4_pair(sb, db);
                  else
                    tc_cp_32x128b_warpx4(sb, db);
                }
              }
              // MMA k (K = 64, scale blocks 2k and 2k + 1) reads word k / 2
              // at byte 2 (k % 2)
#pragma unroll
              for (int k = 0; k < 4; ++k) {
                const uint32_t accum = (kb != kb0 || k != 0) ? 1u : 0u;
                const uint32_t id = idesc_mxf4(kTileM, BN, 2u * (k & 1));
                const uint32_t sa = sfa_t + 4 * (k >> 1);
                const uint32_t sb = sfb_t + (k >> 1) * 4 * L::kSfBlocksB;
                if (CG == 2)
                  tc_mma_mxf4_pair(d_tmem, da0 + 2 * k, db0 + 2 * k, id, sa, sb, accum);
                else
                  tc_mma_mxf4(d_tmem, da0 + 2 * k, db0 + 2 * k, id, sa, sb, accum);
              }
              sf_buf ^= 1;
            } else {
#pragma unroll
              for (int k = 0; k < kBlockK / 16; ++k) {
                const uint64_t da = da0 + 2 * k, db = db0 + 2 * k;
                const uint32_t accum = (kb != kb0 || k != 0) ? 1u : 0u;
                if (CG == 2)
                  tc_mma_f16_pair(d_tmem, da, db, idesc, accum);
                else
                  tc_mma_f16(d_tmem, da, db, idesc, accum);
              }
            }
            if (CG == 2)
              tc_commit_pair_multicast(&empty_bar[stage], 0x3);
            else
              tc_commit(&empty_bar[stage]);
            if (++stage == Stages) {
              stage = 0;
              phase ^= 1;
            }
          }
          if (!ok) break;
          if (CG == 2)
            tc_commit_pair_multicast(&tmem_full[acc], 0x3);
          else
            tc_commit(&tmem_full[acc]);
          if (++acc == 2) {
            acc = 0;
            acc_phase ^= 1;
          }
        }
      }
      if (!ok) {
        *abort_flag = 1;
        // Wait for the MMAs already issued before the tensor memory is freed.
        if (CG == 2)
          tc_commit_pair(drain_bar);
        else
          tc_commit(drain_bar);
        mbar_wait(drain_bar, 0, p.timeout_ns, p.status);
      }
    }
  } else if (kMx && (warp == 2 || warp == 3)) {
    // ------------------------------------------------------------ scale images
    // The images of K-block pair kp (stages of K blocks 2 kp and 2 kp + 1 of
    // a tile) are built by warp 2 (once it has allocated the tensor memory)
    // for even pair numbers and warp 3 for odd ones, each walking the ring
    // as the MMA thread does.  When the pair's scale bytes have landed (in
    // the first stage's slot) the warp reads them into registers, writes the
    // first stage's images and reports them on the even CTA's barrier; once
    // the second stage's slot has been freed by the MMA commit of its
    // previous use, it writes that stage's images too, ahead of its operand
    // tiles.  The slot's scale bytes are all in registers before the first
    // report, since the slot may be refilled as soon as that stage is
    // consumed.  Each report follows a proxy fence (generic writes, then
    // the tensor core's reads), which waits about as long as the MMAs of a
    // stage take: two warps share the pairs so that neither falls behind.
    const uint32_t mine = static_cast<uint32_t>(warp - 2);
    uint32_t pair = 0;  // K-block pairs seen so far
    uint32_t sf_loads = 0;  // per slot: parity of the scale loads seen so far
    const uint32_t img0 = CG == 2 ? mapa_shared(smem_addr(&img_ready[0]), 0) : 0u;
    auto report = [&](int st) {
      fence_proxy_async_smem();  // the images, before the tensor core reads them
      __syncwarp();
      if (lane == 0) {
        if (CG == 2 && !leader)
          mbar_arrive_remote(img0 + static_cast<uint32_t>(st * 8));
        else
          mbar_arrive(&img_ready[st]);
      }
    };
    int stage = 0;
    uint32_t phase = 0;
    for (int t = unit0; t < p.num_tiles && ok; t += units) {
      for (int kb = 0; kb < p.num_k_blocks; kb += 2, ++pair) {
        // the pair's stages: `stage` (phase `phase`), then the next slot
        const int st2 = stage + 1 == Stages ? 0 : stage + 1;
        const uint32_t ph2 = stage + 1 == Stages ? phase ^ 1u : phase;
        const bool two = kb + 1 < p.num_k_blocks;
        if ((pair & 1u) == mine) {
          bool ready = mbar_wait_abortable(&sf_full[stage], (sf_loads >> stage) & 1u,
                                           p.timeout_ns, p.status, abort_flag);
          if (!__all_sync(0xffffffffu, ready)) {
            *abort_flag = 1;
            ok = false;
            break;
          }
          MxScaleRows<BN> sr;
          sr.load(smem_sf_rows + stage * L::kSfRowsBytes, lane);
          sr.store(smem_sf + stage * L::kSfBytes, lane, false);
          report(stage);
          if (two) {
            // the slot's previous use is over when the MMA commit of that
            // use has arrived (as the producer waits before refilling it)
            ready = mbar_wait_abortable(&empty_bar[st2], ph2 ^ 1u, p.timeout_ns, p.status,
                                        abort_flag);
            if (!__all_sync(0xffffffffu, ready)) {
              *abort_flag = 1;
              ok = false;
              break;
            }
            sr.store(smem_sf + st2 * L::kSfBytes, lane, true);
            report(st2);
          }
        }
        sf_loads ^= 1u << stage;  // each pair loads once, into its first slot
        stage = two ? (st2 + 1 == Stages ? 0 : st2 + 1) : st2;
        phase = two ? (st2 + 1 == Stages ? ph2 ^ 1u : ph2) : ph2;
      }
    }
  } else if (warp >= kEpiWarp0) {
    // ------------------------------------------------------------ epilogue
    // A warp may only access TMEM lanes 32*(warp % 4) .. +31: warps w and
    // w + 4 share a lane quarter and take one half of the columns each.
    const int ew = (warp - kEpiWarp0) & 3;
    const int half = (warp - kEpiWarp0) >> 2;
    // 32-column chunks of this half: [0, ceil(n/2)) or [ceil(n/2), n)
    constexpr int kChunks = BN / 32;
    const int chunk_lo = half == 0 ? 0 : (kChunks + 1) / 2;
    const int chunk_hi = half == 0 ? (kChunks + 1) / 2 : kChunks;
    const uint32_t empty0 = CG == 2 ? mapa_shared(smem_addr(&tmem_empty[0]), 0) : 0u;
    const uint32_t lane_base = static_cast<uint32_t>(ew * 32) << 16;
    int acc = 0;
    uint32_t acc_phase = 0;
    if (Out == kOutI32) {
      // Exact INT32 (INT8 operands widened to FP16).  Each K chunk of at most
      // 1024 accumulates exact integers in FP32 (|chunk sum| <= 1024 * 2^14 =
      // 2^24); the warp converts them and adds them to running INT32 sums
      // (wrapping mod 2^32), and after the tile's last chunk writes D = alpha
      // * sum + beta * C (mod 2^32) as 32 x 16 INT32 boxes through the
      // staging buffers (or straight from registers without staging).  The
      // two warps of a lane quarter take kCpw 32-column chunks each, their
      // sums in registers (32 per chunk); when BN / 32 is odd the last chunk
      // is split between them, 16 columns each, its sums kept during the
      // tile in the warp's second staging box (sum i of lane l at word 32 i
      // + l: the lanes fall in different banks) and stored first, before
      // the tile's other stores reuse the box: 224 columns keep 96 sum
      // registers a thread, as 192 do, and need no shared memory of their own.
      static_assert(Out != kOutI32 || BN % 32 == 0, "INT32 mode: whole 32-column chunks");
      constexpr int kCpw = BN / 64;  // 32-column chunks per warp in registers
      constexpr bool kSplitLast = BN % 64 == 32;
      const int c_lo = half * kCpw;
      const int wi = warp - kEpiWarp0;
      uint8_t* boxes = smem + L::kOffEpi + wi * 2 * tc::kEpiBoxBytes;
      // this lane's 16 sums of the split chunk, sum i at word 32 i
      uint32_t* xs = reinterpret_cast<uint32_t*>(boxes + tc::kEpiBoxBytes) + lane;
      static_assert(16 * 32 * 4 <= tc::kEpiBoxBytes, "split chunk's sums in one box");
      const uint32_t al = static_cast<uint32_t>(p.alpha_i), be = static_cast<uint32_t>(p.beta_i);
      uint32_t sum[kCpw][32];
      int nstores = 0;  // stores issued; store i goes through box i & 1
      for (int t = unit0; t < p.num_tiles && ok; t += units) {
        int m_blk, n_blk;
        tc::tile_coords(t, p.num_m_blocks, p.num_n_blocks, p.group_m, m_blk, n_blk);
        const int y = m_blk * kTileM + static_cast<int>(rank) * kBlockM + ew * 32;
        if (kSplitLast && p.staged) {
          // the previous tile's stores have read the box the sums go to
          if (lane == 0) bulk_wait_group_read<0>();
          __syncwarp();
        }
        for (int ch = 0; ch < num_chunks; ++ch) {
          const bool ready =
              !aborted(abort_flag) &&
              mbar_wait_sleepy(&tmem_full[acc], acc_phase, p.timeout_ns, p.status, 256);
          if (!__all_sync(0xffffffffu, ready)) {
            *abort_flag = 1;
            ok = false;
            break;
          }
          tc_fence_after_sync();
          const uint32_t tbase = tmem_base + lane_base + static_cast<uint32_t>(acc * BN);
#pragma unroll
          for (int cl = 0; cl < kCpw; ++cl) {
            uint32_t r[32];
            tmem_ld_32cols(tbase + (c_lo + cl) * 32, r);
            tc_wait_ld();
#pragma unroll
            for (int i = 0; i < 32; ++i) {
              const uint32_t v = static_cast<uint32_t>(__float2int_rn(__uint_as_float(r[i])));
              sum[cl][i] = ch == 0 ? v : sum[cl][i] + v;
            }
          }
          if constexpr (kSplitLast) {
            uint32_t r[16];
            tmem_ld_16cols(tbase + 2 * kCpw * 32 + half * 16, r);
            tc_wait_ld();
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              const uint32_t v = static_cast<uint32_t>(__float2int_rn(__uint_as_float(r[i])));
              xs[i * 32] = ch == 0 ? v : xs[i * 32] + v;
            }
          }
          tc_fence_before_sync();
          if (CG == 2)
            mbar_arrive_cluster(empty0 + static_cast<uint32_t>(acc * 8));
          else
            mbar_arrive(&tmem_empty[acc]);
          if (++acc == 2) {
            acc = 0;
            acc_phase ^= 1;
          }
        }
        if (!ok) break;
        const int row = y + lane;
        const int32_t* crow = static_cast<const int32_t*>(p.C) + static_cast<int64_t>(row) * p.ldc;
        // D's 16 columns from x: o = alpha * sums (+ beta * C), stored
        auto emit = [&](int x, uint32_t (&o)[16]) {
          if (x >= p.N || y >= p.M) return;  // warp-uniform: the box is wholly outside D
          if (be != 0u && row < p.M) {
            if (x + 16 <= p.N && (p.ldc & 3) == 0 &&
                (reinterpret_cast<uintptr_t>(p.C) & 15) == 0) {
#pragma unroll
              for (int q = 0; q < 4; ++q) {
                const uint4 c = *reinterpret_cast<const uint4*>(crow + x + q * 4);
                o[q * 4 + 0] += be * c.x;
                o[q * 4 + 1] += be * c.y;
                o[q * 4 + 2] += be * c.z;
                o[q * 4 + 3] += be * c.w;
              }
            } else {
#pragma unroll
              for (int i = 0; i < 16; ++i)
                if (x + i < p.N) o[i] += be * static_cast<uint32_t>(crow[x + i]);
            }
          }
          if (p.staged) {
            uint8_t* box = boxes + (nstores & 1) * tc::kEpiBoxBytes;
            if (lane == 0) bulk_wait_group_read<1>();  // box's previous store has read it
            __syncwarp();
#pragma unroll
            for (int q = 0; q < 4; ++q)
              *reinterpret_cast<uint4*>(box + tc::epi_box_offset(lane, q)) =
                  make_uint4(o[q * 4], o[q * 4 + 1], o[q * 4 + 2], o[q * 4 + 3]);
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
              tma_store_2d(&tmap_d, box, x, y);
              bulk_commit_group();
            }
            ++nstores;
          } else if (row < p.M) {
            int32_t* drow = static_cast<int32_t*>(p.D) + static_cast<int64_t>(row) * p.ldd;
#pragma unroll
            for (int i = 0; i < 16; ++i)
              if (x + i < p.N) drow[x + i] = static_cast<int32_t>(o[i]);
          }
        };
        if constexpr (kSplitLast) {
          // first, so that its sums are read before a store reuses their box
          uint32_t o[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) o[i] = al * xs[i * 32];
          __syncwarp();
          emit(n_blk * BN + 2 * kCpw * 32 + half * 16, o);
        }
#pragma unroll
        for (int cl = 0; cl < kCpw; ++cl) {
#pragma unroll
          for (int hh = 0; hh < 2; ++hh) {
            uint32_t o[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) o[i] = al * sum[cl][hh * 16 + i];
            emit(n_blk * BN + (c_lo + cl) * 32 + hh * 16, o);
          }
        }
      }
      if (lane == 0) bulk_wait_group<0>();  // stores end before the CTA does
      __syncwarp();
    } else if (p.staged) {
      // Staged epilogue.  The warp's chunks of the works that write D form one
      // stream: chunk j of the stream is chunk k of the warp's share of one
      // tile and goes through box j & 1 of its two boxes.  C of chunks 0 and
      // 1 is loaded by the producer; lane 0 loads C of chunk j + 2 as soon as
      // chunk j's store has read its box, so it arrives while the warp
      // finishes chunk j + 1 or, across tiles, during the next main loop.
      // Tile coordinates are worked out once per work (a second cursor runs
      // two chunks ahead over the works that write D, for the C loads).
      // Reading chunk j + 1's accumulator columns while chunk j is converted
      // was measured and not kept: it took the registers to the 168 limit
      // and the FP16 2048^3 and W4A16 M = 2048 GEMMs 5-7% slower.
      //
      // Stream-K: a work that stores a partial (sk_writer) copies the warp's
      // accumulator region to its slot, then raises its flag; the work that
      // finishes a split tile waits for the flags of the tile's later pieces
      // and adds their partials, in piece order, before the epilogue.
      const int wi = warp - kEpiWarp0;
      uint8_t* boxes = smem + L::kOffEpi + wi * 2 * tc::kEpiBoxBytes;
      uint64_t* cbar = epi_bar + wi * 2;
      const bool has_c = p.epi.beta != 0.0f;
      const uint64_t pol_c = policy_evict_first();
      const int n_mine = chunk_hi - chunk_lo;
      const int row_off = static_cast<int>(rank) * kBlockM + ew * 32;
      // stream-K: the value of this launch's flags
      const unsigned flag_val = SK ? *reinterpret_cast<volatile unsigned*>(sk.sync) + 1u : 0u;
      // The warp's region of partial slot (tile, piece): its 32 rows x its
      // half of the columns, stored as float4 (k * 8 + q) * 32 + lane for
      // columns 4q .. 4q + 3 of chunk k of the lane's row, so that each
      // store and load of the warp covers 512 contiguous bytes.
      auto sk_region = [&](const Work& w, int piece) {
        const int64_t slot =
            static_cast<int64_t>(w.t - sk.dp_tiles) * (sk.max_pieces - 1) + (piece - 1);
        const int region = ((static_cast<int>(rank) * 4 + ew) * 2 + half);
        return reinterpret_cast<float4*>(sk.partial + slot * kTileM * BN) +
               static_cast<int64_t>(region) * (BN / 2) * 8;
      };
      auto sk_flag = [&](const Work& w, int piece) {
        const int64_t slot =
            static_cast<int64_t>(w.t - sk.dp_tiles) * (sk.max_pieces - 1) + (piece - 1);
        return sk.sync + 2 + (slot * CG + rank) * kEpiWarps + wi;
      };
      // A position in the warp's works: the work, chunk k of the warp's share
      // of its tile, the share's first D column x0 and the warp's first D row y.
      struct Cursor {
        WorkWalk w;
        Work wk;
        bool valid;
        int k, x0, y;
      };
      // moves q to the unit's next work (outputs_only: the next that writes D)
      auto seek = [&](Cursor& q, bool outputs_only) {
        bool v = walk_next<SK>(q.w, p, sk, unit0, units, q.wk);
        while (SK && v && outputs_only && sk_writer(q.wk))
          v = walk_next<SK>(q.w, p, sk, unit0, units, q.wk);
        q.valid = v;
        q.k = 0;
        if (v) {
          int mb, nb;
          tc::tile_coords(q.wk.t, p.num_m_blocks, p.num_n_blocks, p.group_m, mb, nb);
          q.x0 = nb * BN + chunk_lo * 32;
          q.y = mb * kTileM + row_off;
        }
      };
      auto advance = [&](Cursor& q) {
        if (++q.k == n_mine) seek(q, true);
      };
      auto live_at = [&](const Cursor& q) {
        return q.valid && q.x0 + q.k * 32 < p.N && q.y < p.M;
      };
      uint32_t c_phase = 0;    // bit b: parity of box b's next C arrival
      uint32_t c_pending = 0;  // bit b: a C load into box b not yet waited for
      bool prev_stored = false;
      Cursor ldc;  // the next chunk whose C is to be requested
      ldc.w = walk_start<SK>(sk, unit0);
      seek(ldc, true);
      for (int jj = 0; jj < 2; ++jj) {  // chunks 0 and 1: requested by the producer
        if (has_c && live_at(ldc)) c_pending |= 1u << jj;
        advance(ldc);
      }
      // Requests C of the chunk at `ldc` (stream index jl) into box jl & 1.
      auto load_c = [&](int jl) {
        if (has_c && live_at(ldc)) {
          const int b = jl & 1;
          c_pending |= 1u << b;
          if (lane == 0) {
            bulk_wait_group_read<0>();  // the store that last used the box has read it
            const int x = ldc.x0 + ldc.k * 32;
            mbar_arrive_expect_tx(&cbar[b], tc::kEpiBoxBytes);
            tma_load_2d(&tmap_c, &cbar[b], boxes + b * tc::kEpiBoxBytes, x, ldc.y, pol_c);
            if (ldc.k == 0)  // the tile's later chunks into L2 ahead of their loads
              for (int k = 2; k < n_mine; ++k)
                if (x + k * 32 < p.N) tma_prefetch_l2_2d(&tmap_c, x + k * 32, ldc.y);
          }
        }
        advance(ldc);
      };
      int j = 0;
      Cursor cur;
      cur.w = walk_start<SK>(sk, unit0);
      seek(cur, false);
      while (cur.valid && ok) {
        const bool ready =
            !aborted(abort_flag) &&
            mbar_wait_sleepy(&tmem_full[acc], acc_phase, p.timeout_ns, p.status, 256);
        if (!__all_sync(0xffffffffu, ready)) {
          *abort_flag = 1;
          ok = false;
          break;
        }
        tc_fence_after_sync();
        const uint32_t tbase =
            tmem_base + lane_base + static_cast<uint32_t>(acc * BN + chunk_lo * 32);
        const bool row_live = cur.y < p.M;
        if (SK && sk_writer(cur.wk)) {
          // the whole region (rows and columns past D included), in stores
          // that stay in L2; then every lane's stores before the flag
          float4* dst = sk_region(cur.wk, cur.wk.piece) + lane;
#pragma unroll 1
          for (int k = 0; k < n_mine; ++k) {
            uint32_t r[32];
            tmem_ld_32cols(tbase + k * 32, r);
            tc_wait_ld();
#pragma unroll
            for (int q = 0; q < 8; ++q)
              __stcg(dst + (k * 8 + q) * 32,
                     make_float4(__uint_as_float(r[4 * q]), __uint_as_float(r[4 * q + 1]),
                                 __uint_as_float(r[4 * q + 2]), __uint_as_float(r[4 * q + 3])));
          }
          __threadfence();
          __syncwarp();
          if (lane == 0) st_release_gpu(sk_flag(cur.wk, cur.wk.piece), flag_val);
        } else {
          if (SK && cur.wk.pieces > 1) {
            // every lane acquires the flags itself before reading partials
            bool got = true;
            for (int q = 1; q < cur.wk.pieces && got; ++q)
              got = wait_flag_eq(sk_flag(cur.wk, q), flag_val, p.timeout_ns, p.status);
            if (!__all_sync(0xffffffffu, got)) {
              *abort_flag = 1;
              ok = false;
              break;
            }
            // the first chunk's partials into L1 (after the acquire: current)
            for (int q = 1; q < cur.wk.pieces; ++q) prefetch_l1(sk_region(cur.wk, q) + lane * 8);
          }
#pragma unroll 1
          for (int k = 0; k < n_mine; ++k) {
            uint32_t r[32];
            const int b = j & 1;
            uint8_t* box = boxes + b * tc::kEpiBoxBytes;
            const int x = cur.x0 + k * 32;
            const bool live = row_live && x < p.N;
            if (live) {
              tmem_ld_32cols(tbase + k * 32, r);
              bool got = true;
              if (has_c) {
                got = mbar_wait(&cbar[b], (c_phase >> b) & 1u, p.timeout_ns, p.status);
                if (got) {
                  c_phase ^= 1u << b;
                  c_pending &= ~(1u << b);
                }
              } else {
                // box b was last read by the store of chunk j - 2
                if (lane == 0) {
                  if (prev_stored)
                    bulk_wait_group_read<1>();
                  else
                    bulk_wait_group_read<0>();
                }
                __syncwarp();
              }
              got = __all_sync(0xffffffffu, got);
              tc_wait_ld();
              if (!got) {
                *abort_flag = 1;
                ok = false;
                break;
              }
              if (SK && cur.wk.pieces > 1) {
                for (int q = 1; q < cur.wk.pieces; ++q) {
                  const float4* src = sk_region(cur.wk, q) + k * 8 * 32 + lane;
                  // the next chunk's 4 KB: one 128-byte line per lane
                  if (k + 1 < n_mine) prefetch_l1(src - lane + 8 * 32 + lane * 8);
#pragma unroll
                  for (int i = 0; i < 8; ++i) {
                    const float4 v = __ldca(src + i * 32);
                    r[4 * i] = __float_as_uint(__uint_as_float(r[4 * i]) + v.x);
                    r[4 * i + 1] = __float_as_uint(__uint_as_float(r[4 * i + 1]) + v.y);
                    r[4 * i + 2] = __float_as_uint(__uint_as_float(r[4 * i + 2]) + v.z);
                    r[4 * i + 3] = __float_as_uint(__uint_as_float(r[4 * i + 3]) + v.w);
                  }
                }
              }
              tc::epilogue_f16_box(r, box, lane, x, p.N, p.epi, prog, p.bias, has_c);
              fence_proxy_async_smem();
              __syncwarp();
              if (lane == 0) {
                tma_store_2d(&tmap_d, box, x, cur.y);
                bulk_commit_group();
              }
            }
            prev_stored = live;
            load_c(j + 2);
            ++j;
          }
        }
        if (!ok) break;
        tc_fence_before_sync();
        if (CG == 2)
          mbar_arrive_cluster(empty0 + static_cast<uint32_t>(acc * 8));
        else
          mbar_arrive(&tmem_empty[acc]);
        if (++acc == 2) {
          acc = 0;
          acc_phase ^= 1;
        }
        seek(cur, false);
      }
      // Copies into and out of the boxes end before the CTA does.
      if (lane == 0) {
        for (int b = 0; b < 2; ++b)
          if (c_pending & (1u << b))
            mbar_wait(&cbar[b], (c_phase >> b) & 1u, p.timeout_ns, p.status);
        bulk_wait_group<0>();
      }
      __syncwarp();
    }
    for (int t = unit0; t < p.num_tiles && ok && Out == kOutF16 && !SK && !p.staged; t += units) {
      int m_blk, n_blk;
      tc::tile_coords(t, p.num_m_blocks, p.num_n_blocks, p.group_m, m_blk, n_blk);
      const int row = m_blk * kTileM + static_cast<int>(rank) * kBlockM + ew * 32 + lane;
      for (int ch = 0; ch < num_chunks; ++ch) {
        if (aborted(abort_flag) ||
            !mbar_wait_sleepy(&tmem_full[acc], acc_phase, p.timeout_ns, p.status, 256)) {
          *abort_flag = 1;
          ok = false;
          break;
        }
        tc_fence_after_sync();
        const uint32_t tbase = tmem_base + lane_base + static_cast<uint32_t>(acc * BN);
#pragma unroll 1
        for (int c = chunk_lo; c < chunk_hi; ++c) {
          uint32_t r[32];
          tmem_ld_32cols(tbase + c * 32, r);
          tc_wait_ld();
          const int col0 = n_blk * BN + c * 32;
          if (col0 < p.N)
            tc::epilogue_f16_chunk(r, row, col0, p.M, p.N, p.epi, prog,
                                   static_cast<const __half*>(p.C), p.ldc,
                                   static_cast<__half*>(p.D), p.ldd, p.bias);
        }
        tc_fence_before_sync();
        if (CG == 2)
          mbar_arrive_cluster(empty0 + static_cast<uint32_t>(acc * 8));
        else
          mbar_arrive(&tmem_empty[acc]);
        if (++acc == 2) {
          acc = 0;
          acc_phase ^= 1;
        }
      }
    }
  }

  tc_fence_before_sync();
  __syncthreads();
  if (CG == 2) {
    if (aborted(abort_flag)) {
      // Copies a peer issued against this pair's barriers may still be in
      // flight after an abort; give them time to land before the pair exits.
      if (threadIdx.x == 0) {
        const uint64_t t0 = global_timer_ns();
        while (global_timer_ns() - t0 < 100000) sleep_ns(1000);
      }
      __syncthreads();
    }
    cluster_sync();  // the peer no longer reads this CTA's shared memory or barriers
  }
  if (warp == 2) {
    tc_fence_after_sync();
    if (CG == 2)
      tmem_dealloc_pair<kTmemCols>(tmem_base);
    else
      tmem_dealloc<kTmemCols>(tmem_base);
  }
  if (SK && threadIdx.x == 0) {
    // The last CTA to finish (aborted or not) advances the epoch: the next
    // launch's flags take the next value.
    __threadfence();
    if (atomicAdd(sk.sync + 1, 1u) == gridDim.x - 1) {
      sk.sync[1] = 0;
      __threadfence();
      atomicAdd(sk.sync, 1u);
    }
  }
}

template <int BN, int Stages, int CG, int Out, int Kind, bool SK = false>
cudaError_t run_tc(const GemmArgs& a, const dg_tile_plan& plan) {
  using L = TcSmem<BN, Stages, CG, Kind>;
  constexpr bool kMx = Kind == kKindMx;
  CUtensorMap ta, tb;
  // A problem with fewer than 128 rows loads only its rows (rounded up to a
  // swizzle atom of 8): TMA is slow on boxes that are mostly out of bounds,
  // and the stale shared-memory rows below only feed accumulator rows >= M,
  // which the epilogue never stores.
  const int box_a = (CG == 1 && a.M < kBlockM) ? static_cast<int>((a.M + 7) / 8 * 8) : kBlockM;
  cudaError_t e;
  if (kMx) {
    // packed codes as bytes: K / 2 bytes per row (K even), 128-byte boxes;
    // the zero fill past K / 2 gives code 0 (value 0) to every K past the end
    e = tc::make_map_2d(&ta, CU_TENSOR_MAP_DATA_TYPE_UINT8, a.A, a.M, a.K / 2, a.lda / 2, box_a,
                        128, CU_TENSOR_MAP_SWIZZLE_128B);
    if (e != cudaSuccess) return e;
    e = tc::make_map_2d(&tb, CU_TENSOR_MAP_DATA_TYPE_UINT8, a.B, a.N, a.K / 2, a.ldb / 2,
                        L::kRowsB, 128, CU_TENSOR_MAP_SWIZZLE_128B);
  } else {
    e = tc::make_f16_kmajor_map(&ta, a.A, a.M, a.K, a.lda, box_a);
    if (e != cudaSuccess) return e;
    e = tc::make_f16_kmajor_map(&tb, a.B, a.N, a.K, a.ldb, L::kRowsB);
  }
  if (e != cudaSuccess) return e;
  // The staged epilogue moves D (and FP16 C) as boxes of 64-byte rows, which
  // needs 16-byte aligned rows (ld % 8 == 0 for FP16, ld % 4 == 0 for INT32)
  // and bases; other layouts store straight from registers.  The INT32 mode
  // reads C with plain loads.
  const int64_t vec = Out == kOutF16 ? 8 : 4;
  const bool c_tma = Out == kOutF16 && a.beta != 0.0f;
  // An int8 D (output quantization) takes the direct path.
  const bool staged = !(a.epi & kEpiOutI8) && a.ldd % vec == 0 &&
                      (reinterpret_cast<uintptr_t>(a.D) & 15) == 0 &&
                      (!c_tma || (a.ldc % vec == 0 && (reinterpret_cast<uintptr_t>(a.C) & 15) == 0));
  CUtensorMap tc_map = ta, td_map = ta;  // copies of a map the kernel does not use
  CUtensorMap tsfa_map = ta, tsfb_map = ta;
  if (kMx) {
    // the row-major scale bytes: boxes of 16 bytes (two stages' scales) by
    // 128 rows of A or BN rows of B (rows start on 16-byte boundaries)
    const int64_t nblk = (a.K + 31) / 32;
    e = tc::make_map_2d(&tsfa_map, CU_TENSOR_MAP_DATA_TYPE_UINT8, a.scale_a, a.M, nblk, a.lds_a,
                        kBlockM, 16, CU_TENSOR_MAP_SWIZZLE_NONE);
    if (e != cudaSuccess) return e;
    e = tc::make_map_2d(&tsfb_map, CU_TENSOR_MAP_DATA_TYPE_UINT8, a.scale_b, a.N, nblk, a.lds_b,
                        BN, 16, CU_TENSOR_MAP_SWIZZLE_NONE);
    if (e != cudaSuccess) return e;
  }
  if (staged) {
    e = Out == kOutF16 ? tc::make_f16_epi_map(&td_map, a.D, a.M, a.N, a.ldd)
                       : tc::make_i32_epi_map(&td_map, a.D, a.M, a.N, a.ldd);
    if (e != cudaSuccess) return e;
    if (c_tma) {
      e = tc::make_f16_epi_map(&tc_map, a.C, a.M, a.N, a.ldc);
      if (e != cudaSuccess) return e;
    }
  }

  TcParams p;
  p.M = static_cast<int>(a.M);
  p.N = static_cast<int>(a.N);
  p.K = static_cast<int>(a.K);
  p.num_m_blocks = static_cast<int>((a.M + kBlockM * CG - 1) / (kBlockM * CG));
  p.num_n_blocks = static_cast<int>((a.N + BN - 1) / BN);
  p.num_tiles = p.num_m_blocks * p.num_n_blocks;
  const int64_t k_per_block = kMx ? 256 : kBlockK;  // K values per stage
  p.num_k_blocks = static_cast<int>((a.K + k_per_block - 1) / k_per_block);
  p.group_m = 16 / CG;
  p.epi = make_epi(a);
  p.C = a.C;
  p.ldc = a.ldc;
  p.D = a.D;
  p.ldd = a.ldd;
  p.bias = static_cast<const __half*>(a.bias);
  p.alpha_i = static_cast<int32_t>(a.alpha);
  p.beta_i = static_cast<int32_t>(a.beta);
  p.status = a.status;
  p.timeout_ns = a.timeout_ns;
  // bytes one stage brings in: both CTAs' operand tiles, counted on the
  // even CTA's barrier for a pair (MXFP4 scale bytes: on each CTA's own)
  p.stage_tx = static_cast<uint32_t>(CG * (box_a * kBlockK * 2 + L::kTileBytesB));
  p.staged = staged ? 1 : 0;
  p.idesc_ab = a.bf16_ab ? idesc_ab_bf16() : 0u;

  auto kern = gemm_tc_kernel<BN, Stages, CG, Out, Kind, SK>;
  int dev = 0;
  cudaGetDevice(&dev);
  // One shared-memory opt-in and one co-residency query per variant and device.
  static std::atomic<uint64_t> attr_set{0};
  static int max_pairs[64] = {};
  cudaLaunchConfig_t cfg = {};
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = L::kLaunchBytes;
  cfg.stream = a.stream;
  cudaLaunchAttribute attr[2];
  cfg.attrs = attr;
  cfg.numAttrs = 0;
  if (CG == 2) {
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
  }
  e = once_per_device(attr_set, dev, [&]() {
    cudaError_t r =
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::kLaunchBytes);
    if (r != cudaSuccess) return r;
    if (CG == 2) {
      // Pairs that fit at once: a persistent grid must not exceed it.
      int n = 0;
      cfg.gridDim = dim3(static_cast<unsigned>(a.sm_count & ~1));
      if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess || n < 1) {
        cudaGetLastError();
        n = a.sm_count / 2;
      }
      max_pairs[dev & 63] = n;
    }
    return cudaSuccess;
  });
  if (e != cudaSuccess) return e;
  // grid: CTAs (pairs x 2 when CG == 2), never more units than tiles
  int units = plan.grid > 0 ? plan.grid / CG : a.sm_count / CG;
  if (CG == 2 && units > max_pairs[dev & 63]) units = max_pairs[dev & 63];
  if (units > p.num_tiles && !SK) units = p.num_tiles;
  // Stream-K CTAs wait for one another: every one must be resident at once
  // (one CTA per SM: the shared memory of a CTA exceeds half an SM's)
  if (SK && CG == 1 && units > a.sm_count) units = a.sm_count;
  if (units < 1) units = 1;
  SkParams sk{p.num_tiles, 0, 0, 1, nullptr, nullptr};
  if (SK) {
    // Stream-K needs the staged epilogue; a problem without ragged work (or
    // another layout) runs the data-parallel kernel of the same tile.
    const SkSplit sp = stream_k_split(p.num_tiles, p.num_k_blocks, units);
    if (!staged || sp.sk_tiles == 0) return run_tc<BN, Stages, CG, Out, Kind, false>(a, plan);
    const int64_t slots = sp.sk_tiles * (sp.max_pieces - 1);
    float* partial = nullptr;
    unsigned* sync = nullptr;
    if (get_sk_workspace(dev, a.stream, std::max<int64_t>(1, slots * kBlockM * CG * BN),
                         2 + slots * CG * kEpiWarps, &partial, &sync) != DG_OK)
      return cudaErrorMemoryAllocation;
    sk.dp_tiles = static_cast<int>(sp.dp_tiles);
    sk.sk_units = sp.sk_units;
    sk.sk_iters = sp.sk_iters;
    sk.max_pieces = sp.max_pieces;
    sk.partial = partial;
    sk.sync = sync;
    // every unit with a whole tile or a range
    const int64_t busy = std::max<int64_t>(std::min<int64_t>(sp.dp_tiles, units), sp.sk_units);
    units = static_cast<int>(std::max<int64_t>(1, busy));
  }
  cfg.gridDim = dim3(static_cast<unsigned>(units * CG));
  // Programmatic dependent launch: this grid's CTAs may start (and set up
  // barriers and tensor memory) while the previous kernel in the stream
  // drains; the kernel waits for that kernel before touching global memory.
  attr[cfg.numAttrs].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[cfg.numAttrs].val.programmaticStreamSerializationAllowed = 1;
  cfg.numAttrs += 1;
  e = cudaLaunchKernelEx(&cfg, kern, ta, tb, tc_map, td_map, tsfa_map, tsfb_map, p,
                         make_program(a), sk);
  count_launches(1);
  return e;
}

template <int BN, int Stages, int CG, int Out, int Kind = kKind16, bool SK = false>
int regs_of() {
  static std::atomic<int> slot{-1};
  return kernel_regs(gemm_tc_kernel<BN, Stages, CG, Out, Kind, SK>, slot);
}

}  // namespace

int tc_kernel_regs(int n_tile, int stages, int cta_group, bool exact_i32) {
  if (exact_i32) {
    if (n_tile == 224 && cta_group == 2 && stages == 6) return regs_of<224, 6, 2, kOutI32>();
    if (n_tile == 192 && cta_group == 2 && stages == 6) return regs_of<192, 6, 2, kOutI32>();
    if (n_tile == 128 && cta_group == 1 && stages == 6) return regs_of<128, 6, 1, kOutI32>();
    return 0;
  }
  if (cta_group == 2) {
    if (n_tile == 256 && stages == 6) return regs_of<256, 6, 2, kOutF16>();
    if (n_tile == 224 && stages == 6) return regs_of<224, 6, 2, kOutF16>();
    if (n_tile == 192 && stages == 6) return regs_of<192, 6, 2, kOutF16>();
    if (n_tile == 128 && stages == 8) return regs_of<128, 8, 2, kOutF16>();
    return 0;
  }
  if (n_tile == 256 && stages == 4) return regs_of<256, 4, 1, kOutF16>();
  if (n_tile == 128 && stages == 6) return regs_of<128, 6, 1, kOutF16>();
  if (n_tile == 64 && stages == 8) return regs_of<64, 8, 1, kOutF16>();
  return 0;
}

int tc_streamk_kernel_regs(int n_tile, int stages, int cta_group) {
  if (n_tile == 256 && stages == 6 && cta_group == 2) return regs_of<256, 6, 2, kOutF16, kKind16, true>();
  if (n_tile == 128 && stages == 6 && cta_group == 1) return regs_of<128, 6, 1, kOutF16, kKind16, true>();
  return 0;
}

int mx_kernel_regs(int n_tile, int stages, int cta_group) {
  if (cta_group == 2) {
    if (n_tile == 224 && stages == 5) return regs_of<224, 5, 2, kOutF16, kKindMx>();
    if (n_tile == 192 && stages == 5) return regs_of<192, 5, 2, kOutF16, kKindMx>();
    return 0;
  }
  if (n_tile == 224 && stages == 3) return regs_of<224, 3, 1, kOutF16, kKindMx>();
  if (n_tile == 128 && stages == 5) return regs_of<128, 5, 1, kOutF16, kKindMx>();
  return 0;
}

// Tile shapes compiled into the library; the planner only proposes these.
// `a` holds FP16 operands (the caller's, or widened copies) or, with
// a.bf16_ab, BF16 ones (widened MXFP4); a.exact_i32 selects the exact INT32
// output of widened INT8 operands.
cudaError_t launch_tc(const GemmArgs& a, const dg_tile_plan& plan) {
  if (a.exact_i32) {
    // 224 columns: 19 x 16 = 304 pair tiles at 4096^2, four whole waves of
    // 76 pairs (192 columns: 352 tiles, 4.63 waves)
    if (plan.n_tile == 224 && plan.cta_group == 2 && plan.stages == 6)
      return run_tc<224, 6, 2, kOutI32, kKind16>(a, plan);
    if (plan.n_tile == 192 && plan.cta_group == 2 && plan.stages == 6)
      return run_tc<192, 6, 2, kOutI32, kKind16>(a, plan);
    if (plan.n_tile == 128 && plan.cta_group == 1 && plan.stages == 6)
      return run_tc<128, 6, 1, kOutI32, kKind16>(a, plan);
    return cudaErrorNotSupported;
  }
  if (plan.cta_group == 2) {
    if (plan.n_tile == 256 && plan.stages == 6) return run_tc<256, 6, 2, kOutF16, kKind16>(a, plan);
    // 224 columns: 19 column tiles cover N = 4096 (the last one partly), so a
    // 4096^2 output is 16 x 19 = 304 pair tiles, four whole waves of 76 pairs
    if (plan.n_tile == 224 && plan.stages == 6) return run_tc<224, 6, 2, kOutF16, kKind16>(a, plan);
    // 192 columns: N = 8960 is 47 column tiles, so M = 2048 gives 376 pair
    // tiles, 4.95 waves of 76 pairs (256 columns: 280 tiles, 3.68 waves)
    if (plan.n_tile == 192 && plan.stages == 6) return run_tc<192, 6, 2, kOutF16, kKind16>(a, plan);
    if (plan.n_tile == 128 && plan.stages == 8) return run_tc<128, 8, 2, kOutF16, kKind16>(a, plan);
    return cudaErrorNotSupported;
  }
  switch (plan.n_tile) {
    case 256:
      if (plan.stages == 4) return run_tc<256, 4, 1, kOutF16, kKind16>(a, plan);
      break;
    case 128:
      if (plan.stages == 6) return run_tc<128, 6, 1, kOutF16, kKind16>(a, plan);
      break;
    case 64:
      if (plan.stages == 8) return run_tc<64, 8, 1, kOutF16, kKind16>(a, plan);
      break;
  }
  return cudaErrorNotSupported;
}

// Stream-K tiles (FP16 x FP16): whole tiles first, then the rest of the
// tiles' K blocks in even ranges over the units.
cudaError_t launch_tc_streamk(const GemmArgs& a, const dg_tile_plan& plan) {
  if (a.exact_i32 || a.bf16_ab) return cudaErrorNotSupported;
  if (plan.n_tile == 256 && plan.stages == 6 && plan.cta_group == 2)
    return run_tc<256, 6, 2, kOutF16, kKind16, true>(a, plan);
  if (plan.n_tile == 128 && plan.stages == 6 && plan.cta_group == 1)
    return run_tc<128, 6, 1, kOutF16, kKind16, true>(a, plan);
  return cudaErrorNotSupported;
}

// MXFP4 tiles on the block-scaled MMA: `a` holds packed codes (K even) and
// row-major scale bytes whose rows start on 16-byte boundaries.
cudaError_t launch_tc_mx(const GemmArgs& a, const dg_tile_plan& plan) {
  if (plan.cta_group == 2) {
    if (plan.n_tile == 224 && plan.stages == 5) return run_tc<224, 5, 2, kOutF16, kKindMx>(a, plan);
    if (plan.n_tile == 192 && plan.stages == 5) return run_tc<192, 5, 2, kOutF16, kKindMx>(a, plan);
    return cudaErrorNotSupported;
  }
  if (plan.n_tile == 224 && plan.stages == 3) return run_tc<224, 3, 1, kOutF16, kKindMx>(a, plan);
  if (plan.n_tile == 128 && plan.stages == 5) return run_tc<128, 5, 1, kOutF16, kKindMx>(a, plan);
  return cudaErrorNotSupported;
}

}  // namespace dg
