// pkd_decode_tc.cuh -- decode attention with both products on the fifth-
// generation tensor cores (tcgen05), scores and output accumulator held in
// tensor memory.
//
// Work split: one CTA per (sequence b, kv head g, partition j, query chunk),
// the split-K decomposition of the partitioned decode in the review
// "Accelerating LLM Inference Throughput via Asynchronous KV Cache
// Prefetching" (section 3.4).  The CTA's tile rows are (query token r / G,
// head r % G) for up to kTcRows rows: every query head of the group and up to
// kTcRows / G query tokens share one pass over the partition's K and V, so a
// multi-token query (speculative verification) reads the cache once per
// chunk of kTcRows / G tokens rather than once per 16 / G.  Two variations of
// the split: the RUNS build takes R consecutive partitions of its (b, g) in
// one stream of tiles and writes each one's partial (short partitions would
// each pay the CTA's fill); and a grid walked longest first whose last round
// would be short reads pieces coded whole sequence / first half / second half
// (tail_split), a half being its own partition of tail_half_partition(L).
//
// Roles (five warps over fp16 caches, six over E4M3):
//   fp16: warps 2    producers: 3-D tensor copies of the partition's K (warp 2)
//   and 4, lane 0    and V (warp 4) tiles of TN tokens (the 128-byte swizzled
//                    layout the MMA descriptors read) into two rings, NSK
//                    stages for K and NSV for V, one mbarrier per stage with
//                    the transaction count of its copies.  A K stage is free
//                    again once S of its tile is computed, a V stage only
//                    after P.V.  One thread per ring: a tile's eight copies
//                    take about a thousand cycles to issue from one thread,
//                    which bounded the tile rate when one thread fed both
//                    rings.  The block ids of a tile are read one issue ahead.
//                    Optionally, tiles beyond the K ring are prefetched into
//                    L2 (cp.async.bulk.prefetch.L2).
//   E4M3: warp 5,    copy issuer: the copies of both rings (four per tile and
//   lane 0           cache at block size 16), each as soon as its stage is
//                    free; the bytes land in a stage's first 8 KiB behind a
//                    landing barrier.  The block ids of a K tile are kept for
//                    its V copy.
//   E4M3: warps 2    wideners of the K (warp 2) and V (warp 3) rings: once a
//   and 3            tile's bytes landed, the whole warp widens them in place
//                    to the fp16 layout the MMAs read and arrives on the
//                    stage's full barrier.  A warp that both issued and
//                    widened was busy for about 70% of a tile period, and its
//                    conversions delayed the next copies.
//   warp 3 (fp16)    MMA issuer: S = Q K^T (M = 128 rows, N = TN tokens,
//   or 4 (E4M3),     K = head_dim) into one of two S buffers in tensor memory,
//   lane 0           then, once the softmax has written P over those S
//                    columns, O += P V (M = 128, N = head_dim, K = TN tokens;
//                    A read from tensor memory) into O in tensor memory;
//                    completion is committed to mbarriers.  It polls both
//                    conditions and issues whichever is ready first: S of the
//                    next tile as soon as its K landed and its S buffer is
//                    free (P.V of the tile two back completed), P.V as soon as
//                    P is written, so the tensor cores overlap the softmax and
//                    neither stage is held behind the other.
//   warps 0-1        softmax, one thread per tile row (tensor-memory lane):
//                    the row of S into registers, mask, online softmax in the
//                    log2 domain with a lazy running maximum (the output is
//                    rescaled in tensor memory only when the maximum grows by
//                    more than kLazyTau), P rounded to fp16 and stored as
//                    fp16 pairs over the tile's S columns (the A operand of
//                    P.V, so no shared memory holds P and the K ring gets a
//                    third stage), and at the end O / l to the output or the
//                    unnormalised partial for the split-K merge.
// The MMAs run M = 128 with the rows past kTcRows reading whatever follows
// Q in shared memory: those accumulator rows, and the P rows made from them,
// are never read, and each output row depends on its own A row only.
//
// The causal rule of multi-token queries is the one of the mma.sync path:
// query jq sits at position L - q_len + jq and sees the tokens before and at
// its position.  Tokens past the CTA's range (the last tile) or in a block
// with a bad id get p = 0, and their V rows are zeroed before P.V so that
// whatever the stage held cannot turn 0 * V into NaN.
//
// Every mbarrier wait is bounded (timeout_ns); a role that gives up records
// kErrTimeout and raises a flag the others poll, the producer waits for the
// copies in flight, the issuer for the MMAs in flight, and tensor memory is
// freed by the warp that allocated it after a final barrier.
#pragma once
#include <cstdint>
#include <cuda.h>
#include <cuda_fp16.h>
#include "pkd_decode_mma.cuh"
#include "pkd_tc.cuh"

namespace pkd {

constexpr int kTcRows = 64;  // query rows per CTA (query tokens x group heads)
constexpr uint32_t kErrLayout = 4u;  // dynamic shared memory not 1024-byte aligned

// Query tokens per CTA of the tcgen05 kernel for group size G.
constexpr int tc_query_chunk(int G) { return kTcRows / G; }

// KVB: bytes per K/V element in the caches (2: fp16; 1: E4M3 bytes, widened
// to fp16 in shared memory by the widening warps before the MMAs read them).
// HD: head_dim, 128 (two 64-dim halves per row) or 64 (one; fp16 only).
template <int BS, int KVB = 2, int HD = 128>
struct TcTraits {
  static_assert(BS == 16 || BS == 32, "block_size");
  static_assert(KVB == 1 || KVB == 2, "fp16 or E4M3 caches");
  static_assert(HD == 64 || HD == 128, "head_dim");
  static_assert(KVB == 2 || HD == 128, "E4M3 rows are widened at head_dim 128 only");
  static constexpr bool F8 = KVB == 1;
  static constexpr int D = HD;
  static constexpr int NH = D / 64;        // 64-dim halves of a row
  static constexpr int ROWS = kTcRows;
  static constexpr int TN = 64;            // tokens per tile
  static constexpr int NBT = TN / BS;      // cache blocks per tile
  static constexpr int NSK = HD == 128 ? 3 : 4;  // K ring stages
  static constexpr int NSV = HD == 128 ? 3 : 5;  // V ring stages
  static constexpr int NPB = 2;            // S buffers in tensor memory, each then holding its tile's P
  static constexpr int ROWB = 128;         // bytes per swizzled row: 64 fp16
  static constexpr int QH = ROWS * ROWB;   // one 64-dim half of Q
  static constexpr int KVH = TN * ROWB;    // one 64-dim half of a K or V tile
  static constexpr int TILE = NH * KVH;    // a K or V tile: its halves
  static constexpr int Q_OFF = 0;
  static constexpr int K_OFF = Q_OFF + NH * QH;
  static constexpr int V_OFF = K_OFF + NSK * TILE;
  static constexpr int MAIN = V_OFF + NSV * TILE;
  static_assert(Q_OFF + (NH - 1) * QH + 128 * ROWB <= MAIN, "the M = 128 operand reads stay inside shared memory");
  static_assert(TN % 16 == 0 && TN / 2 == 32, "P of a row: 32 columns of fp16 pairs, K = 16 tokens per 8");
  // kfull, kempty [NSK]; vfull, vempty [NSV]; sfull[2]; pfull, pfree [NPB]; drain;
  // E4M3: kland [NSK], vland [NSV] (the bytes landed, before widening)
  static constexpr int NBAR = 2 * NSK + 2 * NSV + 2 + 2 * NPB + 1 + (F8 ? NSK + NSV : 0);
  // roles: warps 0-1 softmax; fp16: warp 2 K producer, 3 MMA issuer, 4 V producer;
  // E4M3: warp 2 K widener, 3 V widener, 4 MMA issuer, 5 copy issuer
  static constexpr int W_K = 2;
  static constexpr int W_V = F8 ? 3 : 4;
  static constexpr int W_MMA = F8 ? 4 : 3;
  static constexpr int W_COPY = 5;
  static constexpr int NIDS = 8;  // E4M3: block ids (and bad mask) of the last NIDS K tiles, for their V copies
  // barriers; tensor-memory address, abort flag; vbad [NSV]; E4M3: ids [NIDS][NBT + 1]
  static constexpr int TAIL = NBAR * 8 + 8 + NSV * 4 + (F8 ? NIDS * (NBT + 1) * 4 : 0);
  // No alignment slack: a kernel without static shared memory gets a dynamic
  // window that starts 1024-byte aligned (checked at run time), and two CTAs
  // of 112 KiB fill the SM's 228 KiB with the 1 KiB each reserves.
  static constexpr int SMEM_BYTES = MAIN + ((TAIL + 15) / 16) * 16;
  static constexpr int THREADS = F8 ? 192 : 160;
  static constexpr int MIN_BLOCKS = 2;
  static_assert(MIN_BLOCKS * (SMEM_BYTES + 1024) <= 228 * 1024, "two CTAs per SM");
  // and never three: a third CTA's tensor-memory allocation would wait for one of them to finish
  static_assert(3 * (SMEM_BYTES + 1024) > 228 * 1024, "at most two CTAs per SM");
  static constexpr uint32_t TMEM_COLS = 256;  // O: columns 0-127; S (then P) buffer s: 128 + 64 s
  static constexpr uint32_t IDESC_S = tc_idesc_f16(128, TN, false);
  static constexpr uint32_t IDESC_O = tc_idesc_f16(128, D, true);
};

// RUNS: the build for runs of consecutive partitions per CTA (P.parts_per_cta
// > 1); the other build has one partition per CTA fixed at compile time.
template <int BS, int KVB, int HD, bool RUNS = false>
__global__ void __launch_bounds__(TcTraits<BS, KVB, HD>::THREADS, TcTraits<BS, KVB, HD>::MIN_BLOCKS)
    paged_decode_tc_kernel(const __grid_constant__ CUtensorMap tmap_k, const __grid_constant__ CUtensorMap tmap_v,
                           const DecodeParams P) {
  using T = TcTraits<BS, KVB, HD>;
  constexpr bool F8 = T::F8;
  constexpr int NSK = T::NSK, NSV = T::NSV, NPB = T::NPB, TN = T::TN, D = T::D;
  extern __shared__ __align__(1024) unsigned char smem_tc[];
  unsigned char* smem = smem_tc;
  const uint32_t sbase = smem_u32(smem);
  if (sbase & 1023u) {  // the swizzled operands need 1024-byte aligned groups
    if (threadIdx.x == 0) record_error(P.error_word, kErrLayout);
    return;
  }
  uint64_t* kfull = reinterpret_cast<uint64_t*>(smem + T::MAIN);  // [NSK] a K tile landed
  uint64_t* kempty = kfull + NSK;  // [NSK] S of the tile computed: the K stage is free
  uint64_t* vfull = kempty + NSK;  // [NSV] a V tile landed (with its bad-block mask)
  uint64_t* vempty = vfull + NSV;  // [NSV] P.V of the tile completed: the V stage is free
  uint64_t* sfull = vempty + NSV;  // [2] S of a tile is in tensor memory
  uint64_t* pfull = sfull + 2;     // [NPB] P of a tile is in tensor memory over its S columns
  uint64_t* pfree = pfull + NPB;   // [NPB] P.V of a tile completed (its S/P columns free, O stable)
  uint64_t* drain = pfree + NPB;   // every MMA issued completed
  uint64_t* kland = drain + 1;     // E4M3: [NSK] a K tile's bytes landed
  uint64_t* vland = kland + NSK;   // E4M3: [NSV] a V tile's bytes landed
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1 + (F8 ? NSK + NSV : 0));
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  volatile uint32_t* vbad = reinterpret_cast<volatile uint32_t*>(tmem_slot + 2);  // [NSV]
  int32_t* tile_ids = reinterpret_cast<int32_t*>(tmem_slot + 2 + NSV);            // E4M3: [NIDS][NBT + 1]

  // work item: query chunk fastest, then partition j (a run of R consecutive
  // partitions from j), then (b, g)
  const int G = P.num_q_heads / P.num_kv_heads;
  const int np_grid = P.max_partitions;
  const int R = (RUNS && P.parts_per_cta > 1 && !P.piece_order) ? P.parts_per_cta : 1;
  const int qc = blockIdx.x % P.q_chunks;
  const int rest = blockIdx.x / P.q_chunks;
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  int j, b, g;
  bool half = false;  // a half of a sequence the order split (its own partition size)
  if (P.piece_order) {
    g = rest % P.num_kv_heads;
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const int piece = P.piece_order[rest / P.num_kv_heads];
    if (P.tail_split) {
      if (piece < 0) return;  // a slot past the batch's pieces
      b = piece >> 2;
      j = (piece & 3) == kPieceSecondHalf ? 1 : 0;
      half = (piece & 3) != kPieceWhole;
    } else {
      b = piece / np_grid;
      j = piece % np_grid;
    }
  } else {
    const int nruns = (np_grid + R - 1) / R;
    j = (rest % nruns) * R;
    const int bg = rest / nruns;
    g = bg % P.num_kv_heads;
    b = bg / P.num_kv_heads;
  }
  const int L = row_clamped_len<BS>(P, b);
  const int QL = P.q_len;
  const int jq0 = qc * (T::ROWS / G);         // first query token of this CTA
  const int nq = min(T::ROWS / G, QL - jq0);  // its query tokens (>= 1)
  const int rows = G * nq;                    // tile rows in use
  const int PS = half ? tail_half_partition(L) : P.partition_size;
  const int np_b = min((L + PS - 1) / PS, np_grid);
  const bool final_out = (P.mode == 0) && np_b <= 1;
  const int Hq = P.num_q_heads;
  auto out_row = [&](int rr) { return ((size_t)b * QL + jq0 + rr / G) * Hq + g * G + rr % G; };

  if (L <= 0) {
    if (final_out && j == 0) {
      for (int i = threadIdx.x; i < rows * D; i += blockDim.x)
        P.out[out_row(i / D) * D + i % D] = __float2half_rn(0.f);
    }
    return;
  }
  if (j >= np_b) return;
  // the CTA's partitions [j, j_end); with R > 1 the partition size is a
  // multiple of TN, so every tile lies in one partition, tpp tiles each
  const int j_end = min(j + R, np_b);
  constexpr int kOneRun = 1 << 30;  // tiles per partition when a CTA has one
  const int tpp = RUNS ? (R > 1 ? PS / TN : kOneRun) : kOneRun;

  const int t0 = j * PS;
  // the chunk's last query sees tokens < L - QL + jq0 + nq; nothing past that is read
  const int t1 = min(min(j_end * PS, L), L - QL + jq0 + nq);
  const int ntiles = t1 > t0 ? (t1 - t0 + TN - 1) / TN : 0;
  const int nblk = t1 > t0 ? (t1 - t0 + BS - 1) / BS : 0;
  const int32_t* bt = P.block_tables + (size_t)b * P.max_blocks_per_seq + t0 / BS;
  const int warp = threadIdx.x / 32;
  const int lane = threadIdx.x % 32;
  const int nsw = rows > 32 ? 2 : 1;  // softmax warps

  // ---- producer state (fp16: warp 2, lane 0: K; warp 4, lane 0: V; E4M3: warp 5, lane 0: both)
  const L2Hints l2h = make_l2_hints(P.l2_hints != 0);
  const size_t tile_bytes = (size_t)BS * D * KVB;  // one (block, head) tile
  const size_t block_stride = (size_t)P.num_kv_heads * tile_bytes;
  const char* kbase = reinterpret_cast<const char*>(P.k_cache) + (size_t)g * tile_bytes;
  const char* vbase = reinterpret_cast<const char*>(P.v_cache) + (size_t)g * tile_bytes;
  // the prefetch_distance tiles past the furthest K copy issued are
  // prefetched into L2 (both caches)
  int kissued = 0, vissued = 0;  // tiles whose K / V copies were issued
  int pf_next = 0;
  auto prefetch_upto = [&](int end) {
    for (pf_next = max(pf_next, kissued), end = min(end, ntiles); pf_next < end; ++pf_next) {
#pragma unroll
      for (int kk = 0; kk < T::NBT; ++kk) {
        const int k = pf_next * T::NBT + kk;
        const int pb = k < nblk ? bt[k] : -1;
        if (pb >= 0 && pb < P.num_blocks) {
          prefetch_l2_bulk(kbase + (size_t)pb * block_stride, (uint32_t)tile_bytes, l2h);
          prefetch_l2_bulk(vbase + (size_t)pb * block_stride, (uint32_t)tile_bytes, l2h);
        }
      }
    }
  };
  // the boxes of one tile of one cache into a stage
  auto copy_tile = [&](uint32_t dst, const CUtensorMap* map, uint64_t* bar, const int (&pbs)[T::NBT]) {
#pragma unroll
    for (int kk = 0; kk < T::NBT; ++kk) {
      if (pbs[kk] < 0) continue;
#pragma unroll
      for (int rg = 0; rg < BS / 16; ++rg) {
        const uint32_t row = (kk * BS + 16 * rg) * T::ROWB;
        if constexpr (F8) {
          // E4M3 rows of 128 bytes land in the stage's first 8 KiB, 128-byte swizzled
          tma_load_3d(dst + row, map, bar, 0, g * BS + 16 * rg, pbs[kk], l2h);
        } else {
#pragma unroll
          for (int h = 0; h < T::NH; ++h)
            tma_load_3d(dst + h * T::KVH + row, map, bar, 64 * h, g * BS + 16 * rg, pbs[kk], l2h);
        }
      }
    }
  };
  // Block ids of tile i as stored (-1 past the partition), read one issue
  // ahead of their use so that no copy waits for a block-table read.
  auto load_ids = [&](int i, int (&raw)[T::NBT]) {
#pragma unroll
    for (int kk = 0; kk < T::NBT; ++kk) {
      const int k = i * T::NBT + kk;
      raw[kk] = (i < ntiles && k < nblk) ? bt[k] : -1;
    }
  };
  // The ids of tile i to copy: bad ones (reported once, with the K copy) and
  // those past the partition are skipped (-1); returns the bad-block mask.
  auto check_ids = [&](int i, const int (&raw)[T::NBT], int (&pbs)[T::NBT], bool report) -> uint32_t {
    uint32_t bad = 0;
#pragma unroll
    for (int kk = 0; kk < T::NBT; ++kk) {
      const int k = i * T::NBT + kk;
      int pb = k < nblk ? raw[kk] : -1;
      if (k < nblk && (pb < 0 || pb >= P.num_blocks)) {
        bad |= 1u << kk;
        if (report) record_error(P.error_word, kErrBadBlock);
        pb = -1;
      }
      pbs[kk] = pb;
    }
    return bad;
  };
  auto tile_bytes_of = [&](const int (&pbs)[T::NBT]) {
    uint32_t bytes = 0;
#pragma unroll
    for (int kk = 0; kk < T::NBT; ++kk) bytes += pbs[kk] >= 0 ? BS * D * KVB : 0;  // the block's rows
    return bytes;
  };
  // fp16: issue the copies of tile kissued (K) / vissued (V) into its stage;
  // kraw / vraw hold that tile's block ids.
  int kraw[T::NBT], vraw[T::NBT];
  auto issue_k = [&]() {
    int pbs[T::NBT];
    check_ids(kissued, kraw, pbs, true);
    const int sk = kissued % NSK;
    mbar_arrive_expect_tx(&kfull[sk], tile_bytes_of(pbs));
    copy_tile(sbase + T::K_OFF + sk * T::TILE, &tmap_k, &kfull[sk], pbs);
    ++kissued;
    load_ids(kissued, kraw);
    prefetch_upto(kissued + P.prefetch_distance);
  };
  auto issue_v = [&]() {
    int pbs[T::NBT];
    const uint32_t bad = check_ids(vissued, vraw, pbs, false);
    const int sv = vissued % NSV;
    vbad[sv] = bad;
    mbar_arrive_expect_tx(&vfull[sv], tile_bytes_of(pbs));
    copy_tile(sbase + T::V_OFF + sv * T::TILE, &tmap_v, &vfull[sv], pbs);
    ++vissued;
    load_ids(vissued, vraw);
  };

  // fp16: the first tile's block ids are read before the CTA-wide barrier, so
  // that the first copies do not wait for the block table (2% on 512-token
  // partitions; the E4M3 copy issuer measured 3-6% slower with it).
  if (!F8 && lane == 0) {
    if (warp == T::W_K) load_ids(0, kraw);
    if (warp == T::W_V) load_ids(0, vraw);
  }

  // Barriers are set up before the CTA-wide barrier; the producer starts after
  // it.  (Issuing the first copies from the producer lane before that barrier,
  // to overlap the Q load, measured 13-16% slower on the same GPU: MHA 412
  // against 356 us, GQA 7:1 with q_len 8 908 against 818 us.)
  if (threadIdx.x == 0) {
    prefetch_tensormap(&tmap_k);
    prefetch_tensormap(&tmap_v);
    // E4M3: the full barriers count the 32 lanes of the widening warp
    for (int s = 0; s < NSK; ++s) {
      mbar_init(&kfull[s], F8 ? 32 : 1);
      mbar_init(&kempty[s], 1);
      if (F8) mbar_init(&kland[s], 1);
    }
    for (int s = 0; s < NSV; ++s) {
      mbar_init(&vfull[s], F8 ? 32 : 1);
      mbar_init(&vempty[s], 1);
      if (F8) mbar_init(&vland[s], 1);
    }
    mbar_init(&sfull[0], 1);
    mbar_init(&sfull[1], 1);
    for (int s = 0; s < NPB; ++s) {
      mbar_init(&pfull[s], 32 * nsw);
      mbar_init(&pfree[s], 1);
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_mbarrier_init();
  }
  if (warp == T::W_MMA) {
    tmem_alloc(tmem_slot, T::TMEM_COLS);
    tmem_relinquish();
  }
  if (warp < 2) {
    // Q rows into the two 64-dim halves, 128-byte swizzled; unused rows zero
    const int rr = threadIdx.x;
    const __half* qr = rr < rows ? P.q + out_row(rr) * D : nullptr;
#pragma unroll
    for (int c = 0; c < D / 8; ++c) {
      const uint4 v = qr ? *reinterpret_cast<const uint4*>(qr + 8 * c) : make_uint4(0u, 0u, 0u, 0u);
      *reinterpret_cast<uint4*>(smem + T::Q_OFF + (c / 8) * T::QH + rr * T::ROWB + (((c % 8) ^ (rr % 8)) << 4)) = v;
    }
    fence_proxy_async_smem();  // visible to the tensor cores
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (F8 && warp == T::W_COPY) {
    // ------------------------------------------------------------ copy issuer, E4M3
    // K copies of tile kissued once its stage is free (S of the tile NSK back
    // computed), V copies of tile vissued once its stage is free (P.V of the
    // tile NSV back completed), whichever is possible first.
    if (lane == 0) {
      int raw[T::NBT];
      load_ids(0, raw);
      uint64_t t_idle = 0;
      uint32_t idle_polls = 0;
      bool failed = false;
      while (vissued < ntiles) {
        if (*abort_flag) break;
        bool progress = false;
        if (kissued < ntiles && kissued - vissued < T::NIDS &&
            (kissued < NSK || mbar_test(&kempty[kissued % NSK], ((kissued / NSK) - 1) & 1))) {
          int pbs[T::NBT];
          const uint32_t bad = check_ids(kissued, raw, pbs, true);
          int32_t* ids = tile_ids + (kissued % T::NIDS) * (T::NBT + 1);
#pragma unroll
          for (int kk = 0; kk < T::NBT; ++kk) ids[kk] = pbs[kk];
          ids[T::NBT] = (int32_t)bad;
          const int sk = kissued % NSK;
          mbar_arrive_expect_tx(&kland[sk], tile_bytes_of(pbs));
          copy_tile(sbase + T::K_OFF + sk * T::TILE, &tmap_k, &kland[sk], pbs);
          ++kissued;
          load_ids(kissued, raw);
          prefetch_upto(kissued + P.prefetch_distance);
          progress = true;
        }
        if (vissued < kissued && (vissued < NSV || mbar_test(&vempty[vissued % NSV], ((vissued / NSV) - 1) & 1))) {
          const int32_t* ids = tile_ids + (vissued % T::NIDS) * (T::NBT + 1);
          int pbs[T::NBT];
#pragma unroll
          for (int kk = 0; kk < T::NBT; ++kk) pbs[kk] = ids[kk];
          const int sv = vissued % NSV;
          vbad[sv] = (uint32_t)ids[T::NBT];
          mbar_arrive_expect_tx(&vland[sv], tile_bytes_of(pbs));
          copy_tile(sbase + T::V_OFF + sv * T::TILE, &tmap_v, &vland[sv], pbs);
          ++vissued;
          progress = true;
        }
        if (progress) {
          t_idle = 0;
        } else if ((++idle_polls & 15u) == 0u) {  // nothing to do: give up after timeout_ns without progress
          const uint64_t now = globaltimer_ns();
          if (t_idle == 0) {
            t_idle = now;
          } else if (now - t_idle > P.timeout_ns) {
            failed = true;
            break;
          }
        }
      }
      if (failed) {
        record_error(P.error_word, kErrTimeout);
        *abort_flag = 1;
      }
      if (*abort_flag) {  // let the copies in flight land before the CTA exits
        for (int t = kissued > NSK ? kissued - NSK : 0; t < kissued; ++t)
          mbar_wait_bounded(&kland[t % NSK], (t / NSK) & 1, P.timeout_ns);
        for (int t = vissued > NSV ? vissued - NSV : 0; t < vissued; ++t)
          mbar_wait_bounded(&vland[t % NSV], (t / NSV) & 1, P.timeout_ns);
      }
    }
  } else if (F8 && (warp == T::W_K || warp == T::W_V)) {
    // ------------------------------------------------------------ wideners, E4M3
    // Once a tile's bytes landed, the whole warp widens them in place to the
    // fp16 layout the MMAs read (every lane reads its 16 chunks of the 8 KiB
    // before any lane writes the 16 KiB), then arrives on the tile's full barrier.
    const bool is_k = warp == T::W_K;
    const int ns = is_k ? NSK : NSV;
    uint64_t* land_bar = is_k ? kland : vland;
    uint64_t* full_bar = is_k ? kfull : vfull;
    const uint32_t ring = is_k ? T::K_OFF : T::V_OFF;
    for (int t = 0; t < ntiles; ++t) {
      const int st = t % ns;
      const bool got = !*abort_flag && mbar_wait_bounded(&land_bar[st], (t / ns) & 1, P.timeout_ns);
      if (!__all_sync(0xffffffffu, got)) {
        if (lane == 0) {
          if (!*abort_flag) record_error(P.error_word, kErrTimeout);
          *abort_flag = 1;
        }
        break;
      }
      unsigned char* stg = smem + ring + st * T::TILE;
      uint4 in[16];  // chunk q = lane + 32 k: row q / 8, stored chunk q % 8
#pragma unroll
      for (int k = 0; k < 16; ++k) in[k] = *reinterpret_cast<const uint4*>(stg + 16 * (lane + 32 * k));
      __syncwarp();
#pragma unroll
      for (int k = 0; k < 16; ++k) {
        const int q = lane + 32 * k, r = q >> 3;
        const int j = (q & 7) ^ (r & 7);  // dims 16 j .. 16 j + 15 of row r
        uint4 lo, hi;                     // fp16 dims 16 j .. +7 and 16 j + 8 .. +15
        e4m3x4_to_f16x2x2(in[k].x, lo.x, lo.y);
        e4m3x4_to_f16x2x2(in[k].y, lo.z, lo.w);
        e4m3x4_to_f16x2x2(in[k].z, hi.x, hi.y);
        e4m3x4_to_f16x2x2(in[k].w, hi.z, hi.w);
        const int c0 = 2 * j;  // fp16 chunk (of 16 over both 64-dim halves)
        *reinterpret_cast<uint4*>(stg + (c0 >> 3) * T::KVH + r * T::ROWB + (((c0 & 7) ^ (r & 7)) << 4)) = lo;
        const int c1 = c0 + 1;
        *reinterpret_cast<uint4*>(stg + (c1 >> 3) * T::KVH + r * T::ROWB + (((c1 & 7) ^ (r & 7)) << 4)) = hi;
      }
      fence_proxy_async_smem();  // visible to the tensor cores
      mbar_arrive(&full_bar[st]);
    }
  } else if (!F8 && (warp == T::W_K || warp == T::W_V)) {
    // ------------------------------------------------------------ producers, fp16
    if (lane == 0) {
      const bool is_k = warp == T::W_K;
      const int ns = is_k ? NSK : NSV;
      uint64_t* empty_bar = is_k ? kempty : vempty;
      while ((is_k ? kissued : vissued) < ntiles) {
        if (*abort_flag) break;
        const int i = is_k ? kissued : vissued;
        if (i >= ns && !mbar_wait_bounded(&empty_bar[i % ns], ((i / ns) - 1) & 1, P.timeout_ns)) {
          record_error(P.error_word, kErrTimeout);
          *abort_flag = 1;
          break;
        }
        if (is_k) {
          issue_k();
        } else {
          issue_v();
        }
      }
      if (*abort_flag) {  // let the copies in flight land before the CTA exits
        const int issued = is_k ? kissued : vissued;
        uint64_t* full_bar = is_k ? kfull : vfull;
        for (int k = issued > ns ? issued - ns : 0; k < issued; ++k)
          mbar_wait_bounded(&full_bar[k % ns], (k / ns) & 1, P.timeout_ns);
      }
    }
  } else if (warp == T::W_MMA) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      const uint32_t qs = sbase + T::Q_OFF;
      bool any = false;
      auto issue_qk = [&](int i) -> bool {
        const int sk = i % NSK;
        if (!mbar_wait_bounded(&kfull[sk], (i / NSK) & 1, P.timeout_ns)) return false;
        tc_fence_after();
        const uint32_t ks = sbase + T::K_OFF + sk * T::TILE;
        const uint32_t d = tmem + 128 + 64 * (i & 1);
#pragma unroll
        for (int k = 0; k < D / 16; ++k) {
          const uint32_t off = (k / 4) * T::KVH + (k % 4) * 32;  // 16 dims = 32 bytes of a row
          tc_mma_f16(d, sw128_desc(qs + (k / 4) * T::QH + (k % 4) * 32, 16, 1024), sw128_desc(ks + off, 16, 1024),
                     T::IDESC_S, k > 0 ? 1u : 0u);
        }
        tc_commit(&sfull[i & 1]);
        tc_commit(&kempty[sk]);
        any = true;
        return true;
      };
      // Whichever is ready first: S of tile nq (its K landed, and its S
      // columns are free once P.V of tile nq - 2, which read its P from
      // them, completed), or P.V of tile npv (its P written).  Neither waits
      // behind the other.
      int nq = 0, npv = 0;
      bool ok = true;
      uint64_t t_idle = 0;
      uint32_t idle_polls = 0;
      while (npv < ntiles) {
        if (*abort_flag) {
          ok = false;
          break;
        }
        if (nq < ntiles && nq <= npv + 1 && (nq < NPB || mbar_test(&pfree[nq % NPB], ((nq - NPB) / NPB) & 1)) &&
            mbar_test(&kfull[nq % NSK], (nq / NSK) & 1)) {
          if (!(ok = issue_qk(nq))) break;
          ++nq;
          t_idle = 0;
        } else if (npv < nq && mbar_test(&pfull[npv % NPB], (npv / NPB) & 1)) {
          tc_fence_after();
          const uint32_t vs = sbase + T::V_OFF + (npv % NSV) * T::TILE;
          const uint32_t pa = tmem + 128 + 64 * (npv % NPB);  // P: 8 columns per 16 tokens
#pragma unroll
          for (int k = 0; k < TN / 16; ++k)  // 16 tokens: 8 columns of P, 16 rows of V
            tc_mma_f16_ts(tmem, pa + 8 * k, sw128_desc(vs + k * 16 * T::ROWB, T::KVH, 1024), T::IDESC_O,
                          ((RUNS ? npv % tpp : npv) != 0 || k > 0) ? 1u : 0u);  // a partition's first tile starts O
          tc_commit(&pfree[npv % NPB]);
          tc_commit(&vempty[npv % NSV]);
          ++npv;
          t_idle = 0;
        } else if ((++idle_polls & 15u) == 0u) {
          // nothing ready: give up after timeout_ns without progress (the
          // timer is read on every 16th idle poll only: its read is slow,
          // and it would delay noticing the barrier that completes next)
          const uint64_t now = globaltimer_ns();
          if (t_idle == 0) {
            t_idle = now;
          } else if (now - t_idle > P.timeout_ns) {
            ok = false;
            break;
          }
        }
      }
      if (!ok) {
        record_error(P.error_word, kErrTimeout);
        *abort_flag = 1;
      }
      if (any) {  // every MMA completes before tensor memory is freed
        tc_commit(drain);
        if (!mbar_wait_bounded(drain, 0, P.timeout_ns)) {
          // the output of this CTA cannot be trusted: report it like any other wait that ran out
          record_error(P.error_word, kErrTimeout);
          *abort_flag = 1;
        }
      }
    }
  } else if (warp < nsw) {
    // ------------------------------------------------------------ softmax
    const int rr = threadIdx.x;  // tile row = tensor-memory lane
    const bool live = rr < rows;
    // tokens at or past lim are masked for this row; an unused row takes the
    // last used row's limit, so that the warp takes one path through the mask
    const int lim = min(t1, L - QL + jq0 + (live ? rr : rows - 1) / G + 1);
    const uint32_t tl = tmem + ((uint32_t)(warp * 32) << 16);
    float m = -INFINITY, mt = -INFINITY, l = 0.f;  // running shift, exact maximum, sum of p
    // The result of partition pj: O / l to the output (a sequence of one
    // partition) or the unnormalised partial for the split-K merge; O is read
    // from tensor memory when have_o (whole warp), else zero.
    auto emit = [&](int pj, bool have_o, float em, float emt, float el) {
      const size_t orow = live ? out_row(rr) : 0;
      const size_t pidx = orow * P.max_partitions + pj;
      // el = 0: the query saw no token.  V = code * v_scale for E4M3 caches (1 for fp16)
      const float inv = el > 0.f ? P.v_scale / el : 0.f;
      // partials are relative to the exact maximum emt; O and el to the shift em
      const float f = em == -INFINITY ? 0.f : ex2_approx(em - emt);
      const float fo = f * P.v_scale;
      // once per partition: kept rolled, as is the rescale below, because the
      // kernel's size costs instruction-cache misses in the hot loops
#pragma unroll 1
      for (int c = 0; c < D / 32; ++c) {
        float o[32];
        if (have_o) {
          tmem_ld32(tl + 32 * c, o);
          tmem_ld_wait();
        } else {
#pragma unroll
          for (int e = 0; e < 32; ++e) o[e] = 0.f;
        }
        if (!live) continue;
        if (final_out) {
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            uint4 w;
            w.x = pack_half2(o[8 * q] * inv, o[8 * q + 1] * inv);
            w.y = pack_half2(o[8 * q + 2] * inv, o[8 * q + 3] * inv);
            w.z = pack_half2(o[8 * q + 4] * inv, o[8 * q + 5] * inv);
            w.w = pack_half2(o[8 * q + 6] * inv, o[8 * q + 7] * inv);
            *reinterpret_cast<uint4*>(P.out + orow * D + 32 * c + 8 * q) = w;
          }
        } else {
          float* dst = P.tmp_out + pidx * D + 32 * c;
#pragma unroll
          for (int q = 0; q < 8; ++q)
            *reinterpret_cast<float4*>(dst + 4 * q) =
                make_float4(o[4 * q] * fo, o[4 * q + 1] * fo, o[4 * q + 2] * fo, o[4 * q + 3] * fo);
        }
      }
      if (live && !final_out) {
        P.max_logits[pidx] = emt * 0.69314718055994530942f;  // log2 units -> natural; -inf if empty
        P.exp_sums[pidx] = el * f;
      }
    };
    // Inside a run: the partial of a finished partition (the sequence is split,
    // so never the final output), in a loop kept rolled to keep the kernel's
    // code small
    auto emit_partial = [&](int pj, float em, float emt, float el) {
      const size_t pidx = (live ? out_row(rr) : 0) * P.max_partitions + pj;
      const float fo = (em == -INFINITY ? 0.f : ex2_approx(em - emt)) * P.v_scale;
#pragma unroll 1
      for (int c = 0; c < D / 32; ++c) {
        float o[32];
        tmem_ld32(tl + 32 * c, o);
        tmem_ld_wait();
        if (live) {
          float* dst = P.tmp_out + pidx * D + 32 * c;
#pragma unroll
          for (int q = 0; q < 8; ++q)
            *reinterpret_cast<float4*>(dst + 4 * q) =
                make_float4(o[4 * q] * fo, o[4 * q + 1] * fo, o[4 * q + 2] * fo, o[4 * q + 3] * fo);
        }
      }
      if (live) {
        P.max_logits[pidx] = emt * 0.69314718055994530942f;
        P.exp_sums[pidx] = el * (fo / P.v_scale);
      }
    };
    bool ok = true;
    for (int i = 0; i < ntiles; ++i) {
      const int sv = i % NSV, sb = i & 1;
      // A new partition starts from a fresh state; the previous one's result
      // leaves O below, once this tile's P is written and before it is released
      const bool part_start = RUNS && i > 0 && i % tpp == 0;
      float pm = 0.f, pmt = 0.f, pl = 0.f;
      if (part_start) {
        pm = m;
        pmt = mt;
        pl = l;
        m = -INFINITY;
        mt = -INFINITY;
        l = 0.f;
      }
      ok = __all_sync(0xffffffffu, !*abort_flag && mbar_wait_bounded(&sfull[sb], (i / 2) & 1, P.timeout_ns));
      if (!ok) break;
      tc_fence_after();
      float s[2][32];
      tmem_ld32(tl + 128 + 64 * sb, s[0]);
      tmem_ld32(tl + 128 + 64 * sb + 32, s[1]);
      tmem_ld_wait();
      // the tile's V and its bad-block mask
      ok = __all_sync(0xffffffffu, mbar_wait_bounded(&vfull[sv], (i / NSV) & 1, P.timeout_ns));
      if (!ok) break;
      const uint32_t bad = vbad[sv];
      const int tb = t0 + i * TN;
      const int nv = lim - tb;             // columns this row sees
      const int valid = min(TN, t1 - tb);  // columns holding the CTA's tokens
      // Unmasked tile, scale >= 0: the maximum of the raw scores times the
      // scale is the maximum of the scaled ones, and the scale goes into the
      // exponent's FMA.  Otherwise scale, then mask (-inf), then the maximum.
      const bool raw = nv >= TN && bad == 0 && P.scale_log2 >= 0.f;
      if (!raw) {
#pragma unroll
        for (int e = 0; e < TN; ++e)
          s[e / 32][e % 32] =
              (e < nv && !((bad >> (e / BS)) & 1u)) ? s[e / 32][e % 32] * P.scale_log2 : -INFINITY;
      }
      float mx[8];
#pragma unroll
      for (int a = 0; a < 8; ++a) {
        const float* v = &s[a / 4][(a % 4) * 8];
        mx[a] = fmaxf(fmaxf(fmaxf(v[0], v[1]), fmaxf(v[2], v[3])), fmaxf(fmaxf(v[4], v[5]), fmaxf(v[6], v[7])));
      }
      float tmax = fmaxf(fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])),
                         fmaxf(fmaxf(mx[4], mx[5]), fmaxf(mx[6], mx[7])));
      const float sc = raw ? P.scale_log2 : 1.f;  // the scale still to apply
      if (raw) tmax *= sc;
      mt = fmaxf(mt, tmax);
      const bool rescale = __any_sync(0xffffffffu, tmax > m + kLazyTau);
      float alpha = 1.f;
      if (rescale) {
        const float mn = fmaxf(m, tmax);
        alpha = (mn == -INFINITY) ? 1.f : ex2_approx(m - mn);
        l *= alpha;
        m = mn;
      }
      // a row that has seen no token yet keeps m = -inf: shift by 0 so that
      // its masked scores give p = 0 rather than NaN
      const float mu = m == -INFINITY ? 0.f : m;
      // p = 2^(s * sc - mu), two lanes per packed FMA; the sum in four packed chains
      const float2 sc2 = make_float2(sc, sc), nmu2 = make_float2(-mu, -mu);
      float2 acc[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
      uint32_t pk[TN / 2];  // p as fp16 pairs: tokens 2e (lower half) and 2e + 1
#pragma unroll
      for (int e = 0; e < TN / 2; ++e) {
        const float2 x = ffma2(make_float2(s[e / 16][(2 * e) % 32], s[e / 16][(2 * e + 1) % 32]), sc2, nmu2);
        const float2 pp = make_float2(ex2_approx(x.x), ex2_approx(x.y));
        acc[e % 4] = __fadd2_rn(acc[e % 4], pp);
        pk[e] = pack_half2(pp.x, pp.y);
      }
      const float2 a01 = __fadd2_rn(acc[0], acc[1]), a23 = __fadd2_rn(acc[2], acc[3]);
      const float2 at = __fadd2_rn(a01, a23);
      l += at.x + at.y;
      // O holds the earlier tiles once P.V of the previous one completed: rescale it in place
      if (i > 0 && rescale && !part_start) {
        ok = __all_sync(0xffffffffu,
                        mbar_wait_bounded(&pfree[(i - 1) % NPB], ((i - 1) / NPB) & 1, P.timeout_ns));
        if (!ok) break;
        tc_fence_after();
#pragma unroll 1
        for (int c = 0; c < D / 32; ++c) {
          float o[32];
          tmem_ld32(tl + 32 * c, o);
          tmem_ld_wait();
#pragma unroll
          for (int e = 0; e < 32; ++e) o[e] *= alpha;
          tmem_st32(tl + 32 * c, o);
        }
      }
      // P over this tile's S columns (read into registers above): the A operand of its P.V
      tmem_st32u(tl + 128 + 64 * sb, pk);
      tmem_st_wait();
      if (valid < TN || bad) {
        // V rows that hold no token of the CTA, or a bad block's: p = 0 there,
        // and 0 * NaN would not be 0
        unsigned char* vt = smem + T::V_OFF + sv * T::TILE;
        for (int x = threadIdx.x; x < T::NH * TN * 8; x += 32 * nsw) {
          const int h = x / (TN * 8), r = (x / 8) % TN, c = x % 8;
          if (r >= valid || ((bad >> (r / BS)) & 1u))
            *reinterpret_cast<uint4*>(vt + h * T::KVH + r * T::ROWB + c * 16) = make_uint4(0u, 0u, 0u, 0u);
        }
        fence_proxy_async_smem();  // the zeroed V rows visible to the tensor cores
      }
      if (part_start) {
        // the previous partition is complete once P.V of its last tile is; this
        // tile's P.V (released below) starts O anew
        ok = __all_sync(0xffffffffu,
                        mbar_wait_bounded(&pfree[(i - 1) % NPB], ((i - 1) / NPB) & 1, P.timeout_ns));
        if (!ok) break;
        tc_fence_after();
        emit_partial(j + i / tpp - 1, pm, pmt, pl);
      }
      tc_fence_before();  // our tensor-memory reads and writes ordered before the arrive
      mbar_arrive(&pfull[i % NPB]);
    }
    if (ok && ntiles > 0)
      ok = __all_sync(0xffffffffu, mbar_wait_bounded(&pfree[(ntiles - 1) % NPB], ((ntiles - 1) / NPB) & 1,
                                                     P.timeout_ns));
    if (!ok) {
      if (lane == 0) record_error(P.error_word, kErrTimeout);
      *abort_flag = 1;
    } else {
      tc_fence_after();
      if constexpr (RUNS) {
        // the partition of the last tile, then the CTA's partitions past it
        // (none of the chunk's queries sees their tokens): empty partials
        const int jl = ntiles > 0 ? j + (ntiles - 1) / tpp : j - 1;
        for (int pj = max(jl, j); pj < j_end; ++pj) {
          const bool last = pj == jl;  // else no query of the chunk sees its tokens
          emit(pj, last, last ? m : -INFINITY, last ? mt : -INFINITY, last ? l : 0.f);
        }
      } else {
        emit(j, ntiles > 0, m, mt, l);
      }
    }
  }

  // tensor memory is freed once every warp is done with it
  tc_fence_before();
  __syncthreads();
  if (warp == T::W_MMA) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, T::TMEM_COLS);
  }
}

}  // namespace pkd
