// pkd_api.cu -- the C ABI of libpaged_decode.so (declared in paged_decode.h):
// argument checks, the split-K policy, workspace layout and launches.
#include <algorithm>
#include <atomic>
#include <cmath>
#include <mutex>
#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

#include "../../include/paged_decode.h"
#include "pkd_aux.cuh"
#include "pkd_decode_mma.cuh"
#include "pkd_launch.cuh"
#include "pkd_tc_launch.h"

namespace {

constexpr unsigned long long kWaitBudgetNs = 100ull * 1000ull * 1000ull;  // 100 ms per bounded wait
constexpr int kMinAutoPartition = 512;
constexpr int kMaxAutoPartition = 2048;
constexpr int kMinSmallGridPartition = 128;    // the shortest partition of the one-wave rule (auto_partition)
constexpr int kMinSmallGridPartitionTc = 256;  // the same on the tcgen05 path (64-token tiles)
constexpr int kTcRunMaxPartition = 1024;  // tcgen05: partitions up to this long are taken in runs,
constexpr int kTcRunTokens = 4096;        // ... a CTA streaming up to this many tokens of them
constexpr int kTcRunWaves = 4;            // ... while the grid keeps at least this many waves
// The tcgen05 kernel pays a longer fill per CTA (barriers, tensor memory, and
// the first copies' full HBM latency), so it is split less: only below kSplitWaves
// waves whatever the context length, into partitions of up to
// kMaxAutoPartitionTc tokens.  Measured on its multi-token workloads: GQA 7:1
// at 8192 tokens, q_len 8, unsplit 708 against 788 us at 2048-token
// partitions (q_len 4: 703 against 735); GQA 5:1 at 16K-32K tokens, q_len 8,
// 4096-token partitions 545 against 564 at 2048 and 607 unsplit.  Through the
// automatic path (longest first when unsplit): GQA 7:1, q_len 8, 717 against
// 788 us; q_len 4, 709 against 735.
constexpr int kMaxAutoPartitionTc = 8192;
constexpr int kSplitWaves = 2;       // split when the (sequence, kv head) units cover fewer waves than this,
constexpr int kTargetWaves = 6;      // into enough partitions for this many waves;
constexpr int kLongContext = 8192;   // contexts this long split below kTargetWaves waves
constexpr int kOrderMaxWaves = 6;    // unsplit grids below this many waves walk longest first,
constexpr int kOrderMinContext = 1024;  // when their contexts reach this many tokens
constexpr int kTailMinContext = 1024;   // tcgen05: the order splits the tail of contexts this long
constexpr size_t kTailInfoBytes = 256;  // the order's tail record (two int32), after the order
// Single-query E4M3 grids of at least this many waves of four CTAs per SM run
// the four-per-SM build: 2-7% faster there (MHA, GQA 7:1 and 5:1, ragged
// GQA 4:1 at batch 256), while a ragged GQA 4:1 batch of 1024 CTAs, bounded by
// its longest CTAs, measured 6% slower.
constexpr int kWideFp8Waves = 3;

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

int sm_count();
// Whether an E4M3 launch runs the four-per-SM build (single-query grids of
// kWideFp8Waves waves or more of four CTAs per SM).
bool wide_fp8_grid(int kv_fp8, int q_len, long long grid) {
  int sms = sm_count();
  if (sms <= 0) sms = 148;
  return kv_fp8 && q_len == 1 && grid >= (long long)kWideFp8Waves * 4 * sms;
}

size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

struct Shape {
  int num_seqs, num_q_heads, num_kv_heads, head_dim, block_size, num_blocks, max_blocks_per_seq,
      max_context_len;
};

pkd_status check_shape(const Shape& s) {
  if (s.num_seqs < 0 || s.num_q_heads <= 0 || s.num_kv_heads <= 0 || s.head_dim <= 0 ||
      s.block_size <= 0 || s.num_blocks <= 0 || s.max_blocks_per_seq <= 0 || s.max_context_len < 0)
    return PKD_ERR_SHAPE;
  if (s.num_q_heads % s.num_kv_heads != 0) return PKD_ERR_SHAPE;
  const int G = s.num_q_heads / s.num_kv_heads;
  if (G < 1 || G > 8) return PKD_ERR_UNSUPPORTED;
  if (s.head_dim != 64 && s.head_dim != 128) return PKD_ERR_UNSUPPORTED;
  if (s.block_size != 16 && s.block_size != 32) return PKD_ERR_UNSUPPORTED;
  if ((long long)s.max_context_len > (long long)s.max_blocks_per_seq * s.block_size) return PKD_ERR_SHAPE;
  return PKD_OK;
}

int sm_count() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  return n;
}

// ------------------------------------------------------------ L2 prefetch distance
// The default distance (prefetch_distance 0) comes from two bounds.
//  * Capacity, after section 4.2 of the review "Accelerating LLM Inference
//    Throughput via Asynchronous KV Cache Prefetching": a (block, head) tile
//    is M_block = b * d_h * T_block bytes, and one prefetched tile per warp of
//    every CTA in flight occupies M_total = M_block * (N_thread / 32) * H * B
//    of L2 (all H * B CTAs resident there).  Prefetched tiles past the L2
//    size evict one another before use.  Here only resident CTAs prefetch,
//    and each unit of distance is one more block of K and of V per warp, so
//    footprint(d) = resident CTAs * d * warps * 2 * M_block.  On GB300 the
//    prefetched tiles share L2 with the stream's own lines: distances whose
//    footprint passed about an eighth of L2 measured 1-3% slower, a third
//    5-12% (MHA: the staged path at distances 2 and 4, the tensor-core path
//    at 1-3), so the cap is kL2PrefetchFraction of L2.
//  * Need (Little's law): HBM holds its bandwidth only while each SM keeps
//    about (its share of the bandwidth) x (loaded latency) bytes requested
//    ahead of use.  A CUDA-core warp has one 16-row group of K and V in
//    flight; a staged warp keeps its ring's other slots in flight.  The
//    distance is the smallest that reaches the need, and 0 when the ring
//    alone reaches it.  kLoadedLatencyS is 1.5 us: at 64 KiB per SM the
//    CUDA-core path measured 0.7-10% faster with distance 1 than with none
//    (more at higher group sizes, whose longer iterations hold fewer bytes
//    in flight), while the tensor-core path's 96 KiB per SM gained nothing
//    from any distance.
constexpr double kL2PrefetchFraction = 0.125;
constexpr double kLoadedLatencyS = 1.5e-6;
constexpr int kMaxPrefetchDistance = 8;

// How a data path streams K/V: resident CTAs per SM, block streams (warps)
// per CTA, and bytes each CTA keeps requested ahead of use with no L2
// prefetch.  The values restate the kernels' traits (checked below).
struct PathStream {
  int ctas_per_sm;
  int streams;
  long long ahead_bytes;
  bool prefetches;  // the path issues L2 prefetches at all
};

constexpr int clamp_slots(long long s) { return s > 8 ? 8 : (s < 2 ? 2 : (int)s); }
// slots of a staged ring of ring_kib KiB over `streams` streams of slot_bytes each
constexpr int ring_slots(int ring_kib, int streams, long long slot_bytes) {
  return clamp_slots((ring_kib * 1024LL) / (streams * slot_bytes));
}
static_assert(ring_slots(64, 4, 2 * 16 * 128 * 2) == pkd::MmaTraits<128, 16, 7, 1, 2>::SW, "mma ring (fp16)");
static_assert(ring_slots(64, 4, 2 * 16 * 128 * 1) == pkd::MmaTraits<128, 16, 7, 1, 1>::SW, "mma ring (E4M3)");
static_assert(ring_slots(48, 4, 2 * 16 * 128 * 1) == pkd::MmaTraits<128, 16, 1, 1, 1, 4>::SW, "mma ring (4/SM)");
static_assert(ring_slots(96, 4, 2 * 16 * 128 * 2) == pkd::DecodeTraits<128, 16, 1, pkd::kTmaStaged>::SW, "staged");
static_assert(ring_slots(64, 4, 2 * 16 * 128 * 2) == pkd::DecodeTraits<128, 16, 4, pkd::kTmaStaged>::SW, "staged 3/SM");
static_assert(pkd::DecodeTraits<128, 16, 4, pkd::kTmaStaged>::MIN_BLOCKS == 3 &&
              pkd::DecodeTraits<128, 16, 1, pkd::kTmaStaged>::MIN_BLOCKS == 2 &&
              pkd::DecodeTraits<128, 16, 4, pkd::kL2Prefetch>::MIN_BLOCKS == 2 &&
              pkd::WsTraits<128, 16, 7>::MIN_BLOCKS == 2 && pkd::WsTraits<128, 16, 7>::NS == 3 &&
              pkd::WsTraits<128, 16, 7>::SW == 4 && pkd::WsTraits<64, 16, 7>::SW == 8,
              "residency and streams of the CUDA-core kernels");

PathStream path_stream(int path, int D, int G, int kvb, bool wide_fp8) {
  const long long slot = 2LL * 16 * D * kvb;  // one 16-row group of K and of V
  switch (path) {
    case PKD_VARIANT_NO_PREFETCH:
    case PKD_VARIANT_L2_PREFETCH:
      return {2, 4, 4 * slot, path == PKD_VARIANT_L2_PREFETCH};
    case PKD_VARIANT_TMA_STAGED:
      if (G >= pkd::kWsMinGroup) return {2, 3, 3LL * ((D == 128 ? 4 : 8) - 1) * slot, true};
      if (G >= 2 && G <= 5) return {3, 4, 4LL * (ring_slots(64, 4, slot) - 1) * slot, true};
      return {2, 4, 4LL * (ring_slots(96, 4, slot) - 1) * slot, true};
    case PKD_VARIANT_TMA_MMA: {
      const int cps = wide_fp8 ? 4 : 3;
      return {cps, 4, 4LL * (ring_slots(cps >= 4 ? 48 : 64, 4, slot) - 1) * slot, true};
    }
    default:  // the tcgen05 path streams whole 64-token tiles and never prefetches to L2
      return {2, 2, 0, false};
  }
}

struct DeviceNumbers {
  int sms;
  long long l2_bytes;
  double hbm_bytes_per_s;
};

// The current device's SM count, L2 size and nominal HBM bandwidth (2 x
// memory clock x bus width); GB300-like values where a query fails (no GPU).
// Queried once per device and kept: the memory-clock query costs hundreds of
// microseconds, far more than a decode launch, and none of these change.
DeviceNumbers query_device_numbers(int dev) {
  DeviceNumbers n{148, 126LL << 20, 8.0e12};
  int v = 0;
  if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess && v > 0) n.sms = v;
  if (cudaDeviceGetAttribute(&v, cudaDevAttrL2CacheSize, dev) == cudaSuccess && v > 0) n.l2_bytes = v;
  int clk_khz = 0, bus_bits = 0;
  if (cudaDeviceGetAttribute(&clk_khz, cudaDevAttrMemoryClockRate, dev) == cudaSuccess &&
      cudaDeviceGetAttribute(&bus_bits, cudaDevAttrGlobalMemoryBusWidth, dev) == cudaSuccess && clk_khz > 0 &&
      bus_bits > 0)
    n.hbm_bytes_per_s = 2.0 * clk_khz * 1e3 * (bus_bits / 8.0);
  return n;
}

constexpr int kMaxDevices = 64;
std::mutex g_dev_mu;
std::atomic<int> g_dev_ready[kMaxDevices];
DeviceNumbers g_dev_numbers[kMaxDevices];

DeviceNumbers device_numbers() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();  // no device: leave no sticky error behind
    return DeviceNumbers{148, 126LL << 20, 8.0e12};
  }
  if (dev < 0 || dev >= kMaxDevices) return query_device_numbers(dev);
  if (!g_dev_ready[dev].load(std::memory_order_acquire)) {
    std::lock_guard<std::mutex> lock(g_dev_mu);
    if (!g_dev_ready[dev].load(std::memory_order_relaxed)) {
      g_dev_numbers[dev] = query_device_numbers(dev);
      g_dev_ready[dev].store(1, std::memory_order_release);
    }
  }
  return g_dev_numbers[dev];
}

}  // namespace

extern "C" int pkd_l2_prefetch_model(long long resident_ctas, int sm_count, int streams_per_cta,
                                     long long m_block, int tiles_per_step, long long ahead_bytes_per_cta,
                                     long long l2_bytes, double l2_fraction, double hbm_bytes_per_s,
                                     double latency_s, int max_distance, long long* footprint_bytes,
                                     long long* inflight_bytes_per_sm, long long* need_bytes_per_sm) {
  if (resident_ctas < 0 || sm_count <= 0 || streams_per_cta <= 0 || m_block <= 0 || tiles_per_step <= 0 ||
      ahead_bytes_per_cta < 0 || l2_bytes < 0 || !(l2_fraction >= 0.0) || !(hbm_bytes_per_s >= 0.0) ||
      !(latency_s >= 0.0) || max_distance < 0)
    return -2;
  const long long step = (long long)streams_per_cta * tiles_per_step * m_block;  // per CTA per unit of distance
  const long long active = std::max(1LL, std::min<long long>(sm_count, resident_ctas));
  const double ctas_per_sm = (double)resident_ctas / (double)active;
  const double need = hbm_bytes_per_s / (double)active * latency_s;
  int d = 0;
  while (d < max_distance && ctas_per_sm * (double)(ahead_bytes_per_cta + d * step) < need) ++d;
  const double cap = l2_fraction * (double)l2_bytes;
  while (d > 0 && (double)resident_ctas * d * step > cap) --d;
  if (footprint_bytes) *footprint_bytes = resident_ctas * d * step;
  if (inflight_bytes_per_sm) *inflight_bytes_per_sm = (long long)(ctas_per_sm * (double)(ahead_bytes_per_cta + d * step));
  if (need_bytes_per_sm) *need_bytes_per_sm = (long long)need;
  return d;
}

namespace {

// The distance a launch of `grid` CTAs of this data path runs with by
// default: the model above on the device's numbers, and no more blocks
// ahead than a stream of the CTA has after its first (blocks_per_cta over
// the CTA's streams).
int model_prefetch_distance(int path, int D, int BS, int G, int kvb, bool wide_fp8, long long grid,
                            long long blocks_per_cta, const DeviceNumbers& dn) {
  const PathStream ps = path_stream(path, D, G, kvb, wide_fp8);
  if (!ps.prefetches || grid <= 0) return 0;
  const long long resident = std::min<long long>(grid, (long long)ps.ctas_per_sm * dn.sms);
  int d = pkd_l2_prefetch_model(resident, dn.sms, ps.streams, (long long)BS * D * kvb, 2, ps.ahead_bytes,
                                dn.l2_bytes, kL2PrefetchFraction, dn.hbm_bytes_per_s, kLoadedLatencyS,
                                kMaxPrefetchDistance, nullptr, nullptr, nullptr);
  const long long per_stream = (blocks_per_cta + ps.streams - 1) / ps.streams;
  return (int)std::max(0LL, std::min<long long>(d, per_stream - 1));
}

// The L2 prefetch distance a launch runs: none for -1, the model's default
// for 0, otherwise as requested.  tokens_per_cta is the partition (or the
// whole context, unsplit).
int effective_prefetch(int requested, int path, int D, int BS, int G, int kvb, bool wide_fp8, long long grid,
                       int tokens_per_cta) {
  if (requested < 0) return 0;
  if (requested > 0) return requested;
  return model_prefetch_distance(path, D, BS, G, kvb, wide_fp8, grid, (tokens_per_cta + BS - 1) / BS,
                                 device_numbers());
}

// `variant` carries the data path in its low byte and PKD_FLAG_* bits above.
int variant_path(int variant) { return variant & 0xff; }
bool variant_ok(int variant) {
  const int path = variant_path(variant);
  return variant >= 0 && path <= PKD_VARIANT_TCGEN05 &&
         (variant & ~0xff & ~PKD_FLAG_L2_EVICT_HINTS & ~PKD_FLAG_LONGEST_FIRST) == 0;
}

int resolve_variant(int variant) {
  variant = variant_path(variant);
  return variant == PKD_VARIANT_AUTO ? PKD_VARIANT_TMA_MMA : variant;
}

// What the automatic variant runs for one launch: the tensor-core path
// (swizzled tensor copies into a ring, mma for both products), without the
// L2 eviction priorities, which measured neutral on it.  It is the fastest
// path at every point of the batch x context sweep, uniform and ragged.
// (Plain 16-byte loads used to be picked for group size 1 with at most 512
// tokens per CTA and 1-16 CTAs per SM; with three CTAs per SM, and L2
// flushed without dirty lines, the tensor-core path is 0-7% faster there
// too.)
int pick_auto(int variant, int group, long long grid, long long tokens_per_cta) {
  (void)group;
  (void)grid;
  (void)tokens_per_cta;
  if (variant_path(variant) != PKD_VARIANT_AUTO) return variant;
  return PKD_VARIANT_TMA_MMA;
}

// CTAs per SM of the split and order policy's wave unit for a data path and
// group size: the CUDA-core kernels' residency (DecodeTraits::MIN_BLOCKS),
// and two for the tensor-core path, the residency its thresholds were
// measured at (it now runs three or four per SM).
int ctas_per_sm(int variant, int group) {
  return (resolve_variant(variant) == PKD_VARIANT_TMA_STAGED && group >= 2 && group <= 5) ? 3 : 2;
}

// The wave unit of the split and order policy: ctas_per_sm of the data path
// (two CTAs per SM for the tensor-core path, the residency its thresholds
// were measured at) times the SM count.
long long wave_ctas(int variant, int group) {
  int sms = sm_count();
  if (sms <= 0) sms = 148;
  return (long long)sms * ctas_per_sm(variant, group);
}

// Partition size for the automatic split, or -1 for none.  A shape is split
// when its (sequence, kv head) units would give the GPU fewer than
// kSplitWaves waves of resident CTAs, or, for contexts of kLongContext
// tokens and more, fewer than kTargetWaves waves; the partition is then the
// largest power of two (at most kMaxAutoPartition, at least
// kMinAutoPartition tokens) that yields kTargetWaves waves.  Powers of two
// keep partition boundaries aligned with the blocks of every sequence.
// Shorter contexts from two waves up run unsplit: there the merge pass and
// the shorter CTAs cost more than the tail they save (GQA 4:1 at 3.4 waves:
// 168 us unsplit against 180 us at P = 1024), and a ragged batch's tail is
// shortened by walking it longest first instead (auto_order).  Long ones
// split cheaply, and a grid of a few waves of very long CTAs leaves the
// latency-bound E4M3 kernel a costly last wave (GQA 7:1, 8192 tokens: 358
// us at P = 2048 against 394 us unsplit).
int auto_partition(const Shape& s, int variant = PKD_VARIANT_AUTO, int q_chunks = 1) {
  const long long units = (long long)s.num_seqs * s.num_kv_heads * q_chunks;
  if (units <= 0 || s.max_context_len <= kMinAutoPartition) return -1;
  const long long wave = wave_ctas(variant, s.num_q_heads / s.num_kv_heads);
  const bool tc = variant_path(variant) == PKD_VARIANT_TCGEN05;
  const long long split_below = (!tc && s.max_context_len >= kLongContext ? kTargetWaves : kSplitWaves) * wave;
  if (units >= split_below) return -1;
  const long long want = kTargetWaves * wave;
  const long long np = (want + units - 1) / units;
  const long long per = (s.max_context_len + np - 1) / np;
  // Small grids on the tensor-core paths: the target above would want
  // partitions shorter than kMinAutoPartition, and a grid just past one
  // resident wave runs a second, nearly empty one.  The partition is the
  // shortest power of two whose grid still fits one resident wave (three
  // CTAs per SM on the mma.sync path, two on the tcgen05 path).  Measured on
  // batches of 1-16 at 2048 and 8192 tokens, every power-of-two partition:
  //  * mma.sync, single query (MHA, GQA 4:1, GQA 7:1): the fastest split in
  //    15 of 18 shapes and within 6% in the others (the 512-token minimum
  //    was up to 1.34x slower: GQA 4:1, batch 1, 2048 tokens, 12.5 against
  //    16.4 us);
  //  * tcgen05, 8 query tokens (GQA 4:1, GQA 7:1; fp16 and E4M3): the
  //    fastest in 23 of 24 and within 2.5% in the last (the automatic split
  //    before was up to 1.39x slower: GQA 7:1, batch 16, 8192 tokens, E4M3,
  //    57.6 against 80.2 us).
  // Ragged batches gain less: the plan sees only the longest context.
  if (tc || (q_chunks == 1 && resolve_variant(variant) == PKD_VARIANT_TMA_MMA)) {
    int sms = sm_count();
    if (sms <= 0) sms = 148;
    const int G = s.num_q_heads / s.num_kv_heads;
    const long long slots =
        (long long)sms * (tc ? path_stream(PKD_VARIANT_TCGEN05, s.head_dim, G, 2, false).ctas_per_sm
                             : path_stream(PKD_VARIANT_TMA_MMA, s.head_dim, G, 2, false).ctas_per_sm);
    const long long qmax = tc ? kMaxAutoPartitionTc : kMaxAutoPartition;
    for (long long q = tc ? kMinSmallGridPartitionTc : kMinSmallGridPartition; q <= qmax && q < s.max_context_len;
         q *= 2)
      if (units * ((s.max_context_len + q - 1) / q) <= slots) return (int)q;
  }
  const long long pmax = tc ? kMaxAutoPartitionTc : kMaxAutoPartition;
  long long p = kMinAutoPartition;
  // mma.sync: the largest power of two within per; tcgen05: the smallest
  // power of two that covers per (its longer CTAs pay back their fill: GQA 5:1
  // with 8 query tokens at 16K-32K tokens, per = 4088, took 4096-token
  // partitions at 523 us fp16 and 535 us E4M3 against 540 and 572 at 2048)
  while (p * 2 <= pmax && (tc ? p < per : p * 2 <= per)) p *= 2;
  if (p >= s.max_context_len) return -1;
  return (int)p;
}

struct Workspace {
  float* tmp_out;
  float* max_logits;
  float* exp_sums;
  size_t bytes;
};

// Bytes of the longest-first order (one int32 per piece: sequences x partitions
// of the grid) appended to a workspace.
size_t order_bytes(int num_seqs, int np = 1) {
  return round_up((size_t)num_seqs * (size_t)(np > 0 ? np : 1) * sizeof(int32_t), 256);
}

// Partitions of the grid for a partition choice (1 when unsplit).
int grid_partitions(int max_context_len, int P) {
  return (P > 0 && max_context_len > P) ? (max_context_len + P - 1) / P : 1;
}

// Whether the automatic split also walks the batch longest first: an unsplit
// grid of one to kOrderMaxWaves waves, where the last wave's short CTAs
// decide the tail, of contexts long enough that the order kernel's few
// microseconds are paid back.  Lengths of equal sequences leave the order
// harmless (about 1% at 3-7 waves); ragged ones gain up to 1.1x.
bool auto_order(const Shape& s, int variant, int q_chunks, int partition) {
  const long long units = (long long)s.num_seqs * s.num_kv_heads * q_chunks;
  const long long wave = wave_ctas(variant, s.num_q_heads / s.num_kv_heads);
  return partition <= 0 && s.num_seqs >= 2 && s.num_seqs <= pkd::kOrderMaxSeqs &&
         s.max_context_len >= kOrderMinContext && units >= wave && units < kOrderMaxWaves * wave;
}

// Whether a launch walks the sequences longest first: asked for by flag, on
// the tensor-core path, for batches whose lengths fit the order kernel.
bool want_order(int variant, int resolved_path, int num_seqs) {
  return (variant & PKD_FLAG_LONGEST_FIRST) &&
         (resolved_path == PKD_VARIANT_TMA_MMA || resolved_path == PKD_VARIANT_TCGEN05) && num_seqs > 1 &&
         num_seqs <= pkd::kOrderMaxSeqs;
}

Workspace layout(void* base, int num_seqs, int num_q_heads, int head_dim, int np) {
  const size_t rows = (size_t)num_seqs * num_q_heads * np;
  const size_t a = round_up(rows * head_dim * sizeof(float), 256);
  const size_t m = round_up(rows * sizeof(float), 256);
  Workspace w;
  unsigned char* p = static_cast<unsigned char*>(base);
  w.tmp_out = reinterpret_cast<float*>(p);
  w.max_logits = reinterpret_cast<float*>(p ? p + a : nullptr);
  w.exp_sums = reinterpret_cast<float*>(p ? p + a + m : nullptr);
  w.bytes = a + 2 * m;
  return w;
}

// Query chunks per (sequence, kv head) of q_len query tokens: the
// mma.sync kernel serves 16 / G query tokens per CTA (one 16-row tile), the
// tcgen05 kernel kTcRowsPerCta / G.
int query_chunks(int q_len, int G, int path = PKD_VARIANT_TMA_MMA) {
  if (q_len <= 1) return 1;
  const int qc = (path == PKD_VARIANT_TCGEN05 ? pkd::kTcRowsPerCta : 16) / G;
  return (q_len + qc - 1) / qc;
}

// The tensor-core path the automatic variant runs for several query tokens
// per sequence or E4M3 caches.  The mma.sync kernel serves one 16-row tile of
// q_len x G rows per CTA and reads the partition's K and V once per tile; the
// tcgen05 kernel serves up to 64 rows from one read, with S and O in tensor
// memory.  Measured on the full workloads it wins from kTcMinTiles tiles on
// and loses at one, over fp16 caches (GQA 7:1: q_len 8, four tiles, 686
// against 1164 us; q_len 4, two tiles, 682 against 719 us; GQA 4:1, q_len 8,
// two tiles, 200 against 226 us; q_len 4, one tile, 200 against 182 us) and
// over E4M3 caches, whose tiles the tcgen05 kernel widens to fp16 in shared
// memory (GQA 7:1, q_len 8: 661 against 1175 us; GQA 4:1, q_len 8, two tiles:
// 191 against 217 us; the other two-tile shapes within 2%: GQA 7:1, q_len 4,
// 639 against 629 us; GQA 5:1 at 512-token partitions, q_len 4, 763 against
// 749 us).
constexpr int kTcMinTiles = 2;
// head_dim 128, or 64 with fp16 caches (E4M3 rows are widened at 128 only)
bool tc_supports(const Shape& s, int kv_fp8) { return s.head_dim == 128 || (s.head_dim == 64 && !kv_fp8); }
int auto_multi_path(const Shape& s, int q_len, int kv_fp8) {
  const int G = s.num_q_heads / s.num_kv_heads;
  if (tc_supports(s, kv_fp8) && query_chunks(q_len, G, PKD_VARIANT_TMA_MMA) >= kTcMinTiles)
    return PKD_VARIANT_TCGEN05;
  return PKD_VARIANT_TMA_MMA;
}

// Sequences the longest-first order may split in two on the tcgen05 path (0:
// none); the grid has room for all of them.  An unsplit grid whose last round
// of resident CTAs is at most half full runs that round as long as a full
// one: a tcgen05 CTA is bounded by its own chain of hand-offs, so the round's
// few CTAs go no faster.  Splitting the shortest sequences that fill it in two
// gives the round twice the CTAs of half the length; the order kernel splits
// those of them at least half as long as the batch's longest (a ragged batch
// walked longest first already ends on short CTAs).  Measured on GQA 7:1 with
// 8 query tokens, 8192-token contexts: 3 full rounds (batch 228) 567 us fp16
// and 516 us E4M3, with a fourth round of 112 CTAs (batch 256) 676 and 668 us,
// and with its 28 sequences split 672 and 601 us.
int tail_split_seqs(const Shape& s, int q_chunks, int path, bool split, bool order) {
  if (path != PKD_VARIANT_TCGEN05 || split || !order || s.max_context_len < kTailMinContext) return 0;
  int sms = sm_count();
  if (sms <= 0) sms = 148;
  const int G = s.num_q_heads / s.num_kv_heads;
  const long long slots = (long long)sms * path_stream(PKD_VARIANT_TCGEN05, s.head_dim, G, 2, false).ctas_per_sm;
  const long long per_seq = (long long)s.num_kv_heads * q_chunks;
  const long long units = (long long)s.num_seqs * per_seq;
  if (units <= slots) return 0;
  const long long last = units - (units - 1) / slots * slots;  // CTAs of the last round
  if (2 * last > slots) return 0;
  return (int)std::min<long long>(s.num_seqs, (last + per_seq - 1) / per_seq);
}

// Workspace of an automatic call whose plan splits the tail (0 when it does
// not): partials for two partitions per row, the order and its tail record.
size_t tail_split_bytes(const Shape& s, int q_len, int q_chunks, int path, int P) {
  const bool split = P > 0 && s.max_context_len > P;
  const int tail = tail_split_seqs(s, q_chunks, path, split, auto_order(s, path, q_chunks, P));
  if (tail <= 0) return 0;
  return layout(nullptr, s.num_seqs * q_len, s.num_q_heads, s.head_dim, 2).bytes + order_bytes(s.num_seqs + tail) +
         kTailInfoBytes;
}

// The launch plan of one decode call.
struct CallPlan {
  int P;           // tokens per partition (the whole context, rounded up to 32, when unsplit)
  int q_chunks;    // query chunks per (sequence, kv head)
  int np;          // partitions in the grid (1 when unsplit)
  int runs;        // tcgen05: consecutive partitions per CTA (grid = units x ceil(np / runs))
  bool split;      // the split-K merge runs
  long long grid;  // decode CTAs
  int variant;     // the data path it runs, with the PKD_FLAG_* bits that apply
  bool order;      // the batch is walked longest first (when the workspace has room)
  int tail;        // tcgen05, ordered: the shortest sequences the order splits in two (0: none)
};

// The partition, grid, data path and order a call with these arguments runs
// (the shape already checked).
pkd_status plan_call(const Shape& s, int q_len, int variant, int partition_size, int kv_fp8, CallPlan* out) {
  const int G = s.num_q_heads / s.num_kv_heads;
  const int flags = variant & ~0xff;
  const int path = variant_path(variant);
  if (path == PKD_VARIANT_TCGEN05) {
    if (!tc_supports(s, kv_fp8)) return PKD_ERR_UNSUPPORTED;
  } else if (q_len > 1 || kv_fp8) {
    // several query tokens per sequence, or E4M3 caches: the tensor-core paths only
    if (path != PKD_VARIANT_AUTO && path != PKD_VARIANT_TMA_MMA) return PKD_ERR_UNSUPPORTED;
    variant = (path == PKD_VARIANT_AUTO ? auto_multi_path(s, q_len, kv_fp8) : PKD_VARIANT_TMA_MMA) | flags;
  }
  const int q_chunks = query_chunks(q_len, G, variant_path(variant));
  out->q_chunks = q_chunks;
  int P;
  int flags_eff = flags;
  if (partition_size == 0) {
    P = auto_partition(s, variant, q_chunks);
    if (auto_order(s, variant, q_chunks, P)) flags_eff |= PKD_FLAG_LONGEST_FIRST;
  } else if (partition_size == -1) {
    P = -1;
  } else {
    if (partition_size < 0 || partition_size % 32 != 0 || partition_size % s.block_size != 0)
      return PKD_ERR_SHAPE;
    P = partition_size;
  }
  out->split = P > 0 && s.max_context_len > P;
  out->np = out->split ? (s.max_context_len + P - 1) / P : 1;
  if (!out->split) P = s.max_context_len > 0 ? (int)round_up((size_t)s.max_context_len, 32) : 32;
  out->P = P;
  out->grid = (long long)s.num_seqs * s.num_kv_heads * q_chunks * out->np;
  const int v = pick_auto(variant, G, out->grid, P);
  out->order = out->grid > 0 && want_order(flags_eff, variant_path(v), s.num_seqs);
  out->variant = (v & ~PKD_FLAG_LONGEST_FIRST) | (out->order ? PKD_FLAG_LONGEST_FIRST : 0);
  // Runs of partitions on the tcgen05 path: a CTA streams R consecutive
  // partitions of its (sequence, kv head) and writes each one's partial, so
  // short partitions do not each pay the CTA's fill.  R covers up to
  // kTcRunTokens tokens and keeps at least kTcRunWaves waves of CTAs.
  // (Runs of two 2048-token partitions measured slower than one.)
  out->runs = 1;
  if (variant_path(v) == PKD_VARIANT_TCGEN05 && s.head_dim == 128 && out->split && !out->order && P % 64 == 0 &&
      P <= kTcRunMaxPartition) {
    int sms = sm_count();
    if (sms <= 0) sms = 148;
    const long long units = (long long)s.num_seqs * s.num_kv_heads * q_chunks;
    const long long floor_ctas = (long long)kTcRunWaves * sms * path_stream(PKD_VARIANT_TCGEN05, s.head_dim, G, 2, false).ctas_per_sm;
    int r = kTcRunTokens / P;
    while (r > 1 && units * ((out->np + r - 1) / r) < floor_ctas) r /= 2;
    out->runs = r;
    out->grid = units * ((out->np + r - 1) / r);
  }
  out->tail = tail_split_seqs(s, q_chunks, variant_path(v), out->split, out->order);
  if (out->tail > 0) out->grid = ((long long)s.num_seqs + out->tail) * s.num_kv_heads * q_chunks;
  return PKD_OK;
}

pkd_status launch_decode(int variant, int D, int BS, int G, const pkd::DecodeParams& p,
                         long long grid, cudaStream_t stream) {
  if (grid <= 0) return PKD_OK;
  if (grid > 0x7fffffffLL) return PKD_ERR_SHAPE;
  cudaError_t e;
  switch (variant) {
    case PKD_VARIANT_NO_PREFETCH: e = pkd::launch_decode_no_prefetch(D, BS, G, p, grid, stream); break;
    case PKD_VARIANT_L2_PREFETCH: e = pkd::launch_decode_l2_prefetch(D, BS, G, p, grid, stream); break;
    case PKD_VARIANT_TMA_STAGED: e = pkd::launch_decode_tma_staged(D, BS, G, p, grid, stream); break;
    case PKD_VARIANT_TMA_MMA: e = pkd::launch_decode_tma_mma(D, BS, G, p, grid, stream); break;
    case PKD_VARIANT_TCGEN05: e = pkd::launch_decode_tcgen05(D, BS, p, grid, stream); break;
    default: return PKD_ERR_SHAPE;
  }
  return e == cudaSuccess ? PKD_OK : PKD_ERR_LAUNCH;
}

pkd_status launch_reduce(const float* tmp_out, const float* max_logits, const float* exp_sums,
                         const int32_t* context_lens, void* out, int num_seqs, int num_q_heads,
                         int head_dim, int partition_size, int max_num_partitions, int min_merge,
                         cudaStream_t stream, const int32_t* tail_order = nullptr,
                         const int32_t* tail_info = nullptr) {
  const long long rows = (long long)num_seqs * num_q_heads;
  if (rows <= 0) return PKD_OK;
  if (rows > 0x7fffffffLL) return PKD_ERR_SHAPE;
  const long long grid = (rows + pkd::kReduceRowsPerCta - 1) / pkd::kReduceRowsPerCta;
  __half* o = static_cast<__half*>(out);
  // Programmatic dependent launch: the merge may become resident while the
  // decode grid's last CTAs still run; its griddepcontrol.wait holds it until
  // that grid has completed and its partials are visible.
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)grid);
  cfg.blockDim = dim3(32 * pkd::kReduceRowsPerCta);
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t e;
  if (head_dim == 128) {
    e = cudaLaunchKernelEx(&cfg, pkd::paged_decode_reduce_kernel<128>, tmp_out, max_logits, exp_sums,
                           context_lens, o, (int)rows, num_q_heads, partition_size, max_num_partitions, min_merge,
                           tail_order, tail_info);
  } else if (head_dim == 64) {
    e = cudaLaunchKernelEx(&cfg, pkd::paged_decode_reduce_kernel<64>, tmp_out, max_logits, exp_sums,
                           context_lens, o, (int)rows, num_q_heads, partition_size, max_num_partitions, min_merge,
                           tail_order, tail_info);
  } else {
    return PKD_ERR_UNSUPPORTED;
  }
  return e == cudaSuccess && cudaGetLastError() == cudaSuccess ? PKD_OK : PKD_ERR_LAUNCH;
}

pkd_status check_inputs(const void* q, const void* k_cache, const void* v_cache,
                        const int32_t* block_tables, const int32_t* context_lens) {
  if (!q || !k_cache || !v_cache || !block_tables || !context_lens) return PKD_ERR_NULL;
  if (!aligned(q, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16) || !aligned(block_tables, 4) ||
      !aligned(context_lens, 4))
    return PKD_ERR_ALIGN;
  return PKD_OK;
}

}  // namespace

extern "C" {

int pkd_version(void) { return 1 * 10000 + 1 * 100 + 0; }

const char* pkd_status_string(int status) {
  switch (status) {
    case PKD_OK: return "ok";
    case PKD_ERR_NULL: return "a required pointer is NULL";
    case PKD_ERR_SHAPE: return "a size is out of range or inconsistent";
    case PKD_ERR_UNSUPPORTED: return "head_dim, block_size or group size not supported";
    case PKD_ERR_ALIGN: return "a pointer is not suitably aligned";
    case PKD_ERR_WORKSPACE: return "workspace missing or too small";
    case PKD_ERR_LAUNCH: return "CUDA kernel launch failed";
    case PKD_ERR_DEVICE: return "the device reported an error";
    case PKD_ERR_CUDA: return "a CUDA runtime call failed";
    default: return "unknown status";
  }
}

int paged_decode_auto_partition_size(int num_seqs, int num_q_heads, int num_kv_heads, int head_dim,
                                     int block_size, int max_context_len, int variant) {
  Shape s{num_seqs, num_q_heads, num_kv_heads, head_dim, block_size, 1, 1 << 30, max_context_len};
  if (check_shape(s) != PKD_OK) return -2;
  if (!variant_ok(variant)) return -2;
  return auto_partition(s, variant);
}

int paged_decode_auto_variant(int num_seqs, int num_q_heads, int num_kv_heads, int head_dim,
                              int block_size, int max_context_len, int partition_size) {
  Shape s{num_seqs, num_q_heads, num_kv_heads, head_dim, block_size, 1, 1 << 30, max_context_len};
  if (check_shape(s) != PKD_OK || partition_size < -1) return -2;
  CallPlan plan;
  if (plan_call(s, 1, PKD_VARIANT_AUTO, partition_size, 0, &plan) != PKD_OK) return -2;
  return plan.variant;
}

size_t paged_decode_workspace_size(int num_seqs, int num_q_heads, int num_kv_heads, int head_dim,
                                   int block_size, int max_context_len, int partition_size,
                                   int variant) {
  Shape s{num_seqs, num_q_heads, num_kv_heads, head_dim, block_size, 1, 1 << 30, max_context_len};
  if (check_shape(s) != PKD_OK) return 0;
  if (!variant_ok(variant)) return 0;
  int P = partition_size == 0 ? auto_partition(s, variant) : partition_size;
  size_t bytes = 0;
  if (P > 0 && max_context_len > P)
    bytes = layout(nullptr, num_seqs, num_q_heads, head_dim, (max_context_len + P - 1) / P).bytes;
  if ((variant & PKD_FLAG_LONGEST_FIRST) || partition_size == 0)
    bytes += order_bytes(num_seqs, grid_partitions(max_context_len, P));
  if (partition_size == 0 && variant_path(variant) == PKD_VARIANT_TCGEN05)
    bytes = std::max(bytes, tail_split_bytes(s, 1, 1, PKD_VARIANT_TCGEN05, P));
  return bytes;
}

}  // extern "C"

namespace {


// Decode of q_len query tokens per sequence (q_len = 1: single-query decode).
pkd_status decode_impl(const void* q, const void* k_cache, const void* v_cache,
                       const int32_t* block_tables, const int32_t* context_lens, void* out, int num_seqs,
                       int q_len, int num_q_heads, int num_kv_heads, int head_dim, int block_size,
                       int num_blocks, int max_blocks_per_seq, int max_context_len, float scale,
                       int partition_size, int variant, int prefetch_distance, void* workspace,
                       size_t workspace_bytes, int* error_word, cudaStream_t stream, int kv_fp8 = 0,
                       float k_scale = 1.f, float v_scale = 1.f) {
  Shape s{num_seqs, num_q_heads, num_kv_heads, head_dim, block_size, num_blocks, max_blocks_per_seq,
          max_context_len};
  pkd_status st = check_shape(s);
  if (st != PKD_OK) return st;
  if (q_len < 1) return PKD_ERR_SHAPE;
  if (kv_fp8 && !(std::isfinite(k_scale) && std::isfinite(v_scale) && k_scale > 0.f && v_scale > 0.f))
    return PKD_ERR_SHAPE;
  if (num_seqs == 0) return PKD_OK;
  st = check_inputs(q, k_cache, v_cache, block_tables, context_lens);
  if (st != PKD_OK) return st;
  if (!out) return PKD_ERR_NULL;
  if (!aligned(out, 16) || (error_word && !aligned(error_word, 4))) return PKD_ERR_ALIGN;
  if (!std::isfinite(scale)) return PKD_ERR_SHAPE;
  if (!variant_ok(variant)) return PKD_ERR_SHAPE;
  if (prefetch_distance < -1) return PKD_ERR_SHAPE;
  const int G = num_q_heads / num_kv_heads;
  CallPlan plan;
  st = plan_call(s, q_len, variant, partition_size, kv_fp8, &plan);
  if (st != PKD_OK) return st;
  const int P = plan.P, np = plan.np;
  const bool split = plan.split;
  long long grid = plan.grid;
  variant = plan.variant;
  // The tail split keeps its partials (two per row), the order and the
  // order's tail record in the workspace; without room the grid runs unsplit.
  int tail = plan.tail;
  if (tail > 0 && (!workspace || !aligned(workspace, 256) ||
                   workspace_bytes < layout(nullptr, num_seqs * q_len, num_q_heads, head_dim, 2).bytes +
                                         order_bytes(num_seqs + tail) + kTailInfoBytes)) {
    tail = 0;
    grid = (long long)num_seqs * num_kv_heads * plan.q_chunks;
  }

  pkd::DecodeParams p{};
  p.q = static_cast<const __half*>(q);
  p.k_cache = static_cast<const __half*>(k_cache);
  p.v_cache = static_cast<const __half*>(v_cache);
  p.block_tables = block_tables;
  p.context_lens = context_lens;
  p.out = static_cast<__half*>(out);
  p.error_word = error_word;
  p.num_seqs = num_seqs;
  p.num_q_heads = num_q_heads;
  p.num_kv_heads = num_kv_heads;
  p.num_blocks = num_blocks;
  p.max_blocks_per_seq = max_blocks_per_seq;
  p.partition_size = P;
  p.max_partitions = np;
  p.mode = 0;
  p.q_len = q_len;
  p.q_chunks = plan.q_chunks;
  p.parts_per_cta = plan.runs;
  // E4M3 caches: K = code * k_scale enters the scores, V = code * v_scale the output
  p.scale_log2 = scale * (kv_fp8 ? k_scale : 1.f) * 1.4426950408889634f;
  p.v_scale = kv_fp8 ? v_scale : 1.f;
  p.prefetch_distance = effective_prefetch(prefetch_distance, variant_path(variant), head_dim, block_size, G,
                                          kv_fp8 ? 1 : 2, wide_fp8_grid(kv_fp8, q_len, grid), grid, P);
  p.l2_hints = (variant & PKD_FLAG_L2_EVICT_HINTS) ? 1 : 0;
  p.timeout_ns = kWaitBudgetNs;
  size_t used = 0;
  if (split || tail > 0) {
    // partial rows are (sequence, query token, head)
    if (!workspace) return PKD_ERR_WORKSPACE;
    if (!aligned(workspace, 256)) return PKD_ERR_ALIGN;
    Workspace w = layout(workspace, num_seqs * q_len, num_q_heads, head_dim, tail > 0 ? 2 : np);
    if (workspace_bytes < w.bytes) return PKD_ERR_WORKSPACE;
    p.tmp_out = w.tmp_out;
    p.max_logits = w.max_logits;
    p.exp_sums = w.exp_sums;
    used = w.bytes;
  }
  // the order sits after the partials; it only reschedules, so a workspace
  // without room for it runs the plain grid order instead (a tail split's
  // record follows the order)
  int32_t* tail_info = nullptr;
  if (tail > 0) p.max_partitions = 2;
  if (grid > 0 && plan.order && workspace && aligned(workspace, 256) &&
      workspace_bytes >= used + (tail > 0 ? order_bytes(num_seqs + tail) + kTailInfoBytes : order_bytes(num_seqs, np))) {
    unsigned char* at = static_cast<unsigned char*>(workspace) + used;
    int32_t* order = reinterpret_cast<int32_t*>(at);
    if (tail > 0) tail_info = reinterpret_cast<int32_t*>(at + order_bytes(num_seqs + tail));
    pkd::piece_order_kernel<<<(num_seqs + 127) / 128, 128, 0, stream>>>(context_lens, num_seqs, P, np, order, tail,
                                                                        tail_info);
    if (cudaGetLastError() != cudaSuccess) return PKD_ERR_LAUNCH;
    p.piece_order = order;
    p.tail_split = tail > 0 ? 1 : 0;
  }
  if (kv_fp8 && variant_path(variant) == PKD_VARIANT_TCGEN05) {
    if (grid > 0x7fffffffLL) return PKD_ERR_SHAPE;
    const cudaError_t e =
        grid <= 0 ? cudaSuccess : pkd::launch_decode_tcgen05(head_dim, block_size, p, grid, stream, /*kvb=*/1);
    st = e == cudaSuccess ? PKD_OK : PKD_ERR_LAUNCH;
  } else if (kv_fp8) {
    if (grid > 0x7fffffffLL) return PKD_ERR_SHAPE;
    // single-query grids of kWideFp8Waves waves or more of four CTAs per SM
    // run the four-per-SM build
    const bool w4 = wide_fp8_grid(kv_fp8, q_len, grid);
    const cudaError_t e = grid <= 0 ? cudaSuccess
                          : w4      ? pkd::launch_decode_tma_mma_fp8_w4(head_dim, block_size, G, p, grid, stream)
                                    : pkd::launch_decode_tma_mma_fp8(head_dim, block_size, G, p, grid, stream);
    st = e == cudaSuccess ? PKD_OK : PKD_ERR_LAUNCH;
  } else {
    st = launch_decode(variant_path(variant), head_dim, block_size, G, p, grid, stream);
  }
  if (st != PKD_OK || (!split && tail == 0)) return st;
  // the merge sees q_len * Hq rows per sequence; after a tail split, those of
  // the (at most tail) sequences the order split
  if (tail > 0)
    return launch_reduce(p.tmp_out, p.max_logits, p.exp_sums, context_lens, out, tail, q_len * num_q_heads,
                         head_dim, P, 2, /*min_merge=*/1, stream, p.piece_order, tail_info);
  return launch_reduce(p.tmp_out, p.max_logits, p.exp_sums, context_lens, out, num_seqs, q_len * num_q_heads,
                       head_dim, P, np, /*min_merge=*/1, stream);
}

}  // namespace

extern "C" {

pkd_status paged_decode_attention_ex(const void* q, const void* k_cache, const void* v_cache,
                                     const int32_t* block_tables, const int32_t* context_lens,
                                     void* out, int num_seqs, int num_q_heads, int num_kv_heads,
                                     int head_dim, int block_size, int num_blocks,
                                     int max_blocks_per_seq, int max_context_len, float scale,
                                     int partition_size, int variant, int prefetch_distance,
                                     void* workspace, size_t workspace_bytes, int* error_word,
                                     cudaStream_t stream) {
  return decode_impl(q, k_cache, v_cache, block_tables, context_lens, out, num_seqs, 1, num_q_heads,
                     num_kv_heads, head_dim, block_size, num_blocks, max_blocks_per_seq, max_context_len,
                     scale, partition_size, variant, prefetch_distance, workspace, workspace_bytes,
                     error_word, stream);
}

pkd_status paged_decode_attention_multi(const void* q, const void* k_cache, const void* v_cache,
                                        const int32_t* block_tables, const int32_t* context_lens,
                                        void* out, int num_seqs, int q_len, int num_q_heads,
                                        int num_kv_heads, int head_dim, int block_size, int num_blocks,
                                        int max_blocks_per_seq, int max_context_len, float scale,
                                        int partition_size, void* workspace, size_t workspace_bytes,
                                        int* error_word, cudaStream_t stream) {
  return decode_impl(q, k_cache, v_cache, block_tables, context_lens, out, num_seqs, q_len, num_q_heads,
                     num_kv_heads, head_dim, block_size, num_blocks, max_blocks_per_seq, max_context_len,
                     scale, partition_size, PKD_VARIANT_AUTO, 0, workspace, workspace_bytes,
                     error_word, stream);
}

pkd_status paged_decode_attention_multi_ex(const void* q, const void* k_cache, const void* v_cache,
                                           const int32_t* block_tables, const int32_t* context_lens,
                                           void* out, int num_seqs, int q_len, int num_q_heads,
                                           int num_kv_heads, int head_dim, int block_size, int num_blocks,
                                           int max_blocks_per_seq, int max_context_len, float scale,
                                           int partition_size, int variant, void* workspace,
                                           size_t workspace_bytes, int* error_word, cudaStream_t stream) {
  return decode_impl(q, k_cache, v_cache, block_tables, context_lens, out, num_seqs, q_len, num_q_heads,
                     num_kv_heads, head_dim, block_size, num_blocks, max_blocks_per_seq, max_context_len,
                     scale, partition_size, variant, 0, workspace, workspace_bytes, error_word, stream);
}

pkd_status paged_decode_attention_fp8(const void* q, const void* k_cache, const void* v_cache,
                                      const int32_t* block_tables, const int32_t* context_lens, void* out,
                                      int num_seqs, int q_len, int num_q_heads, int num_kv_heads,
                                      int head_dim, int block_size, int num_blocks, int max_blocks_per_seq,
                                      int max_context_len, float scale, float k_scale, float v_scale,
                                      int partition_size, void* workspace, size_t workspace_bytes,
                                      int* error_word, cudaStream_t stream) {
  return decode_impl(q, k_cache, v_cache, block_tables, context_lens, out, num_seqs, q_len, num_q_heads,
                     num_kv_heads, head_dim, block_size, num_blocks, max_blocks_per_seq, max_context_len,
                     scale, partition_size, PKD_VARIANT_AUTO, 0, workspace, workspace_bytes, error_word,
                     stream, 1, k_scale, v_scale);
}

pkd_status paged_decode_attention_fp8_ex(const void* q, const void* k_cache, const void* v_cache,
                                         const int32_t* block_tables, const int32_t* context_lens, void* out,
                                         int num_seqs, int q_len, int num_q_heads, int num_kv_heads,
                                         int head_dim, int block_size, int num_blocks, int max_blocks_per_seq,
                                         int max_context_len, float scale, float k_scale, float v_scale,
                                         int partition_size, int variant, void* workspace, size_t workspace_bytes,
                                         int* error_word, cudaStream_t stream) {
  return decode_impl(q, k_cache, v_cache, block_tables, context_lens, out, num_seqs, q_len, num_q_heads,
                     num_kv_heads, head_dim, block_size, num_blocks, max_blocks_per_seq, max_context_len,
                     scale, partition_size, variant, 0, workspace, workspace_bytes, error_word, stream, 1, k_scale,
                     v_scale);
}

int paged_decode_call_plan(int num_seqs, int q_len, int num_q_heads, int num_kv_heads, int head_dim,
                           int block_size, int max_context_len, int kv_fp8, int partition_size, int variant,
                           int* partition_out, int* longest_first, int* variant_out, long long* grid_out,
                           int* prefetch_distance_out) {
  Shape s{num_seqs, num_q_heads, num_kv_heads, head_dim, block_size, 1, 1 << 30, max_context_len};
  if (check_shape(s) != PKD_OK || q_len < 1 || !variant_ok(variant)) return -2;
  CallPlan plan;
  if (plan_call(s, q_len, variant, partition_size, kv_fp8, &plan) != PKD_OK) return -2;
  if (partition_out) *partition_out = plan.split ? plan.P : -1;
  if (longest_first) *longest_first = plan.order ? 1 : 0;
  if (variant_out) *variant_out = plan.variant;
  if (grid_out) *grid_out = num_seqs == 0 ? 0 : plan.grid;
  if (prefetch_distance_out)
    *prefetch_distance_out =
        num_seqs == 0 ? 0
                      : effective_prefetch(0, variant_path(plan.variant), head_dim, block_size,
                                           num_q_heads / num_kv_heads, kv_fp8 ? 1 : 2,
                                           wide_fp8_grid(kv_fp8, q_len, plan.grid), plan.grid, plan.P);
  if (num_seqs == 0 || plan.grid == 0) return 0;
  return 1 + (plan.split || plan.tail > 0 ? 1 : 0) + (plan.order ? 1 : 0);
}

int paged_decode_prefetch_model(int num_seqs, int q_len, int num_q_heads, int num_kv_heads, int head_dim,
                                int block_size, int max_context_len, int kv_fp8, int partition_size, int variant,
                                int sm_count_, long long l2_bytes, double hbm_bytes_per_s,
                                long long* footprint_bytes, long long* inflight_bytes_per_sm,
                                long long* need_bytes_per_sm) {
  Shape s{num_seqs, num_q_heads, num_kv_heads, head_dim, block_size, 1, 1 << 30, max_context_len};
  if (check_shape(s) != PKD_OK || q_len < 1 || !variant_ok(variant) || sm_count_ <= 0 || l2_bytes <= 0 ||
      !(hbm_bytes_per_s > 0.0))
    return -2;
  CallPlan plan;
  if (plan_call(s, q_len, variant, partition_size, kv_fp8, &plan) != PKD_OK) return -2;
  const int path = variant_path(plan.variant);
  const int G = num_q_heads / num_kv_heads, kvb = kv_fp8 ? 1 : 2;
  const bool wide = kv_fp8 && q_len == 1 && plan.grid >= (long long)kWideFp8Waves * 4 * sm_count_;
  const PathStream ps = path_stream(path, head_dim, G, kvb, wide);
  const long long grid = num_seqs == 0 ? 0 : plan.grid;
  const long long resident = std::min<long long>(grid, (long long)ps.ctas_per_sm * sm_count_);
  int d = pkd_l2_prefetch_model(resident, sm_count_, ps.streams, (long long)block_size * head_dim * kvb, 2,
                                ps.ahead_bytes, l2_bytes, kL2PrefetchFraction, hbm_bytes_per_s, kLoadedLatencyS,
                                ps.prefetches ? kMaxPrefetchDistance : 0, footprint_bytes, inflight_bytes_per_sm,
                                need_bytes_per_sm);
  const long long per_stream = ((plan.P + block_size - 1) / block_size + ps.streams - 1) / ps.streams;
  return (int)std::max(0LL, std::min<long long>(d, per_stream - 1));
}

int paged_decode_auto_plan(int num_seqs, int q_len, int num_q_heads, int num_kv_heads, int head_dim,
                           int block_size, int max_context_len, int kv_fp8, int* partition_size,
                           int* longest_first) {
  return paged_decode_call_plan(num_seqs, q_len, num_q_heads, num_kv_heads, head_dim, block_size,
                                max_context_len, kv_fp8, 0, PKD_VARIANT_AUTO, partition_size, longest_first,
                                nullptr, nullptr, nullptr);
}

size_t paged_decode_multi_workspace_size(int num_seqs, int q_len, int num_q_heads, int num_kv_heads,
                                         int head_dim, int block_size, int max_context_len,
                                         int partition_size) {
  Shape s{num_seqs, num_q_heads, num_kv_heads, head_dim, block_size, 1, 1 << 30, max_context_len};
  if (check_shape(s) != PKD_OK || q_len < 1) return 0;
  // with partition_size 0 the split depends on the path's query chunks: cover
  // both tensor-core paths
  size_t most = 0;
  for (const int path : {PKD_VARIANT_TMA_MMA, PKD_VARIANT_TCGEN05}) {
    if (path == PKD_VARIANT_TCGEN05 && head_dim != 128 && head_dim != 64) continue;
    const int qch = query_chunks(q_len, num_q_heads / num_kv_heads, path);
    const int P = partition_size == 0 ? auto_partition(s, path, qch) : partition_size;
    size_t bytes = 0;
    if (P > 0 && max_context_len > P)
      bytes = layout(nullptr, num_seqs * q_len, num_q_heads, head_dim, (max_context_len + P - 1) / P).bytes;
    if (partition_size == 0)  // the automatic split may order the batch
      bytes += order_bytes(num_seqs, grid_partitions(max_context_len, P));
    most = std::max(most, bytes);
    if (partition_size == 0)  // ... and split its tail
      most = std::max(most, tail_split_bytes(s, q_len, qch, path, P));
  }
  return most;
}

pkd_status paged_decode_attention_host(const void* q, const void* k_cache, const void* v_cache,
                                       const int32_t* block_tables, const int32_t* context_lens, void* out,
                                       void* q_dev, void* k_cache_dev, void* v_cache_dev,
                                       int32_t* block_tables_dev, int32_t* context_lens_dev, void* out_dev,
                                       int num_seqs, int num_q_heads, int num_kv_heads, int head_dim,
                                       int block_size, int num_blocks, int max_blocks_per_seq,
                                       int max_context_len, float scale, int used_blocks_only, void* workspace,
                                       size_t workspace_bytes, int* error_word, cudaStream_t stream) {
  Shape s{num_seqs, num_q_heads, num_kv_heads, head_dim, block_size, num_blocks, max_blocks_per_seq,
          max_context_len};
  pkd_status st = check_shape(s);
  if (st != PKD_OK) return st;
  if (num_seqs == 0) return PKD_OK;
  if (!q || !k_cache || !v_cache || !block_tables || !context_lens || !out || !q_dev || !k_cache_dev ||
      !v_cache_dev || !block_tables_dev || !context_lens_dev || !out_dev)
    return PKD_ERR_NULL;
  if (!aligned(q, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16) || !aligned(out, 16) ||
      !aligned(out_dev, 16) || !aligned(k_cache_dev, 16) || !aligned(v_cache_dev, 16))
    return PKD_ERR_ALIGN;
  const size_t q_bytes = (size_t)num_seqs * num_q_heads * head_dim * 2;
  const size_t block_bytes = (size_t)num_kv_heads * block_size * head_dim * 2;
  const size_t pool_bytes = (size_t)num_blocks * block_bytes;
  const size_t bt_bytes = (size_t)num_seqs * max_blocks_per_seq * sizeof(int32_t);
  const size_t cl_bytes = (size_t)num_seqs * sizeof(int32_t);
  // the small inputs: one copy each
  if (cudaMemcpyAsync(q_dev, q, q_bytes, cudaMemcpyHostToDevice, stream) != cudaSuccess ||
      cudaMemcpyAsync(block_tables_dev, block_tables, bt_bytes, cudaMemcpyHostToDevice, stream) != cudaSuccess ||
      cudaMemcpyAsync(context_lens_dev, context_lens, cl_bytes, cudaMemcpyHostToDevice, stream) != cudaSuccess)
    return PKD_ERR_CUDA;
  // the pools: the used blocks read in place from mapped host memory, or
  // (not mapped, or asked for) one copy of each whole pool
  void* k_map = nullptr;
  void* v_map = nullptr;
  const bool gather = used_blocks_only && cudaHostGetDevicePointer(&k_map, const_cast<void*>(k_cache), 0) == cudaSuccess &&
                      cudaHostGetDevicePointer(&v_map, const_cast<void*>(v_cache), 0) == cudaSuccess;
  if (!gather) {
    (void)cudaGetLastError();  // a failed mapping query is not an error of this call
    if (cudaMemcpyAsync(k_cache_dev, k_cache, pool_bytes, cudaMemcpyHostToDevice, stream) != cudaSuccess ||
        cudaMemcpyAsync(v_cache_dev, v_cache, pool_bytes, cudaMemcpyHostToDevice, stream) != cudaSuccess)
      return PKD_ERR_CUDA;
  } else {
    const int mb = std::min(max_blocks_per_seq, (max_context_len + block_size - 1) / block_size);
    if (mb > 0) {
      if (num_seqs > 65535) return PKD_ERR_SHAPE;
      pkd::gather_used_blocks_kernel<<<dim3((unsigned)mb, (unsigned)num_seqs), 256, 0, stream>>>(
          static_cast<const uint4*>(k_map), static_cast<const uint4*>(v_map), static_cast<uint4*>(k_cache_dev),
          static_cast<uint4*>(v_cache_dev), block_tables_dev, context_lens_dev, max_blocks_per_seq, block_size,
          num_blocks, (long long)(block_bytes / 16), error_word);
      if (cudaGetLastError() != cudaSuccess) return PKD_ERR_LAUNCH;
    }
  }
  st = decode_impl(q_dev, k_cache_dev, v_cache_dev, block_tables_dev, context_lens_dev, out_dev, num_seqs, 1,
                   num_q_heads, num_kv_heads, head_dim, block_size, num_blocks, max_blocks_per_seq,
                   max_context_len, scale, 0, PKD_VARIANT_AUTO, 0, workspace, workspace_bytes, error_word, stream);
  if (st != PKD_OK) return st;
  return cudaMemcpyAsync(out, out_dev, q_bytes, cudaMemcpyDeviceToHost, stream) == cudaSuccess ? PKD_OK
                                                                                               : PKD_ERR_CUDA;
}

pkd_status paged_decode_attention(const void* q, const void* k_cache, const void* v_cache,
                                  const int32_t* block_tables, const int32_t* context_lens, void* out,
                                  int num_seqs, int num_q_heads, int num_kv_heads, int head_dim,
                                  int block_size, int num_blocks, int max_blocks_per_seq,
                                  int max_context_len, float scale, cudaStream_t stream) {
  return paged_decode_attention_ex(q, k_cache, v_cache, block_tables, context_lens, out, num_seqs,
                                   num_q_heads, num_kv_heads, head_dim, block_size, num_blocks,
                                   max_blocks_per_seq, max_context_len, scale, /*partition_size=*/-1,
                                   PKD_VARIANT_AUTO, 0, nullptr, 0, nullptr, stream);
}

pkd_status paged_decode_partitions(const void* q, const void* k_cache, const void* v_cache,
                                   const int32_t* block_tables, const int32_t* context_lens,
                                   int num_seqs, int num_q_heads, int num_kv_heads, int head_dim,
                                   int block_size, int num_blocks, int max_blocks_per_seq,
                                   int max_context_len, float scale, int partition_size,
                                   int variant, int prefetch_distance, float* tmp_out,
                                   float* max_logits, float* exp_sums, int max_num_partitions,
                                   int* error_word, cudaStream_t stream) {
  Shape s{num_seqs, num_q_heads, num_kv_heads, head_dim, block_size, num_blocks, max_blocks_per_seq,
          max_context_len};
  pkd_status st = check_shape(s);
  if (st != PKD_OK) return st;
  if (num_seqs == 0) return PKD_OK;
  st = check_inputs(q, k_cache, v_cache, block_tables, context_lens);
  if (st != PKD_OK) return st;
  if (!tmp_out || !max_logits || !exp_sums) return PKD_ERR_NULL;
  if (!aligned(tmp_out, 16) || !aligned(max_logits, 4) || !aligned(exp_sums, 4) ||
      (error_word && !aligned(error_word, 4)))
    return PKD_ERR_ALIGN;
  if (!std::isfinite(scale)) return PKD_ERR_SHAPE;
  if (!variant_ok(variant) || prefetch_distance < -1)
    return PKD_ERR_SHAPE;
  if (variant_path(variant) == PKD_VARIANT_TCGEN05 && head_dim != 128 && head_dim != 64) return PKD_ERR_UNSUPPORTED;
  if (partition_size <= 0 || partition_size % 32 != 0 || partition_size % block_size != 0)
    return PKD_ERR_SHAPE;
  const int need = (max_context_len + partition_size - 1) / partition_size;
  if (max_num_partitions < (need > 0 ? need : 1)) return PKD_ERR_SHAPE;
  pkd::DecodeParams p{};
  p.q = static_cast<const __half*>(q);
  p.k_cache = static_cast<const __half*>(k_cache);
  p.v_cache = static_cast<const __half*>(v_cache);
  p.block_tables = block_tables;
  p.context_lens = context_lens;
  p.out = nullptr;
  p.tmp_out = tmp_out;
  p.max_logits = max_logits;
  p.exp_sums = exp_sums;
  p.error_word = error_word;
  p.num_seqs = num_seqs;
  p.num_q_heads = num_q_heads;
  p.num_kv_heads = num_kv_heads;
  p.num_blocks = num_blocks;
  p.max_blocks_per_seq = max_blocks_per_seq;
  p.partition_size = partition_size;
  p.max_partitions = max_num_partitions;
  p.mode = 1;
  p.q_len = 1;
  p.q_chunks = 1;
  p.v_scale = 1.f;
  p.scale_log2 = scale * 1.4426950408889634f;
  const int G = num_q_heads / num_kv_heads;
  const long long grid = (long long)num_seqs * num_kv_heads * max_num_partitions;
  variant = pick_auto(variant, G, grid, partition_size);
  p.prefetch_distance = effective_prefetch(prefetch_distance, variant_path(variant), head_dim, block_size, G, 2,
                                           false, grid, partition_size);
  p.l2_hints = (variant & PKD_FLAG_L2_EVICT_HINTS) ? 1 : 0;
  p.timeout_ns = kWaitBudgetNs;
  return launch_decode(variant_path(variant), head_dim, block_size, G, p, grid, stream);
}

pkd_status paged_decode_reduce(const float* tmp_out, const float* max_logits, const float* exp_sums,
                               const int32_t* context_lens, void* out, int num_seqs, int num_q_heads,
                               int head_dim, int partition_size, int max_num_partitions,
                               int min_partitions_to_merge, cudaStream_t stream) {
  if (num_seqs < 0 || num_q_heads <= 0 || partition_size <= 0 || max_num_partitions <= 0 ||
      min_partitions_to_merge < 0)
    return PKD_ERR_SHAPE;
  if (head_dim != 64 && head_dim != 128) return PKD_ERR_UNSUPPORTED;
  if (num_seqs == 0) return PKD_OK;
  if (!tmp_out || !max_logits || !exp_sums || !context_lens || !out) return PKD_ERR_NULL;
  if (!aligned(tmp_out, 4) || !aligned(max_logits, 4) || !aligned(exp_sums, 4) ||
      !aligned(context_lens, 4) || !aligned(out, 2))
    return PKD_ERR_ALIGN;
  return launch_reduce(tmp_out, max_logits, exp_sums, context_lens, out, num_seqs, num_q_heads, head_dim,
                       partition_size, max_num_partitions, min_partitions_to_merge, stream);
}

pkd_status paged_decode_validate_tables(const int32_t* block_tables, const int32_t* context_lens,
                                        int num_seqs, int max_blocks_per_seq, int block_size,
                                        int num_blocks, int* error_word, cudaStream_t stream) {
  if (num_seqs < 0 || max_blocks_per_seq <= 0 || block_size <= 0 || num_blocks <= 0) return PKD_ERR_SHAPE;
  if (num_seqs == 0) return PKD_OK;
  if (!block_tables || !context_lens || !error_word) return PKD_ERR_NULL;
  if (!aligned(block_tables, 4) || !aligned(context_lens, 4) || !aligned(error_word, 4)) return PKD_ERR_ALIGN;
  pkd::validate_tables_kernel<<<num_seqs, 128, 0, stream>>>(block_tables, context_lens, num_seqs,
                                                            max_blocks_per_seq, block_size, num_blocks,
                                                            error_word);
  return cudaGetLastError() == cudaSuccess ? PKD_OK : PKD_ERR_LAUNCH;
}

pkd_status paged_kv_append(const void* k_new, const void* v_new, const int32_t* block_tables,
                           const int32_t* context_lens, void* k_cache, void* v_cache, int num_seqs,
                           int num_kv_heads, int head_dim, int block_size, int num_blocks,
                           int max_blocks_per_seq, int* error_word, cudaStream_t stream) {
  if (num_seqs < 0 || num_kv_heads <= 0 || head_dim <= 0 || head_dim % 8 != 0 || block_size <= 0 ||
      num_blocks <= 0 || max_blocks_per_seq <= 0)
    return PKD_ERR_SHAPE;
  if (num_seqs == 0) return PKD_OK;
  if (!k_new || !v_new || !block_tables || !context_lens || !k_cache || !v_cache) return PKD_ERR_NULL;
  if (!aligned(k_new, 16) || !aligned(v_new, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16) ||
      !aligned(block_tables, 4) || !aligned(context_lens, 4) || (error_word && !aligned(error_word, 4)))
    return PKD_ERR_ALIGN;
  const int chunks = head_dim / 8;
  const long long total = (long long)num_seqs * num_kv_heads * chunks;
  int sms = 152;
  int dev = 0;
  if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const long long want = (total + 255) / 256;
  const int grid = (int)std::min<long long>(want, (long long)sms * 8);
  pkd::paged_kv_append_kernel<<<grid, 256, 0, stream>>>(
      static_cast<const uint4*>(k_new), static_cast<const uint4*>(v_new), block_tables, context_lens,
      static_cast<uint4*>(k_cache), static_cast<uint4*>(v_cache), num_seqs, num_kv_heads, chunks,
      block_size, num_blocks, max_blocks_per_seq, error_word);
  return cudaGetLastError() == cudaSuccess ? PKD_OK : PKD_ERR_LAUNCH;
}

pkd_status paged_kv_append_fp8(const void* k_new, const void* v_new, const int32_t* block_tables,
                               const int32_t* context_lens, void* k_cache, void* v_cache, int num_seqs,
                               int num_kv_heads, int head_dim, int block_size, int num_blocks,
                               int max_blocks_per_seq, float k_scale, float v_scale, int* error_word,
                               cudaStream_t stream) {
  if (num_seqs < 0 || num_kv_heads <= 0 || head_dim <= 0 || head_dim % 16 != 0 || block_size <= 0 ||
      num_blocks <= 0 || max_blocks_per_seq <= 0)
    return PKD_ERR_SHAPE;
  if (!(std::isfinite(k_scale) && std::isfinite(v_scale) && k_scale > 0.f && v_scale > 0.f))
    return PKD_ERR_SHAPE;
  if (num_seqs == 0) return PKD_OK;
  if (!k_new || !v_new || !block_tables || !context_lens || !k_cache || !v_cache) return PKD_ERR_NULL;
  if (!aligned(k_new, 16) || !aligned(v_new, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16) ||
      !aligned(block_tables, 4) || !aligned(context_lens, 4) || (error_word && !aligned(error_word, 4)))
    return PKD_ERR_ALIGN;
  const int chunks = head_dim / 16;  // 16 output bytes per thread
  const long long total = (long long)num_seqs * num_kv_heads * chunks;
  int sms = sm_count();
  if (sms <= 0) sms = 148;
  const int grid = (int)std::min<long long>((total + 255) / 256, (long long)sms * 8);
  pkd::paged_kv_append_fp8_kernel<<<grid, 256, 0, stream>>>(
      static_cast<const uint4*>(k_new), static_cast<const uint4*>(v_new), block_tables, context_lens,
      static_cast<uint4*>(k_cache), static_cast<uint4*>(v_cache), num_seqs, num_kv_heads, chunks, block_size,
      num_blocks, max_blocks_per_seq, k_scale, v_scale, error_word);
  return cudaGetLastError() == cudaSuccess ? PKD_OK : PKD_ERR_LAUNCH;
}

pkd_status pkd_selftest_bounded_wait(int* error_word, unsigned long long budget_ns, cudaStream_t stream) {
  if (!error_word) return PKD_ERR_NULL;
  if (!aligned(error_word, 4)) return PKD_ERR_ALIGN;
  if (budget_ns < 1000ull || budget_ns > kWaitBudgetNs) return PKD_ERR_SHAPE;
  pkd::selftest_bounded_wait_kernel<<<1, 32, 0, stream>>>(error_word, budget_ns);
  return cudaGetLastError() == cudaSuccess ? PKD_OK : PKD_ERR_LAUNCH;
}

pkd_status pkd_read_device_error(int* error_word, unsigned* host_bits, int clear, cudaStream_t stream) {
  if (!error_word || !host_bits) return PKD_ERR_NULL;
  unsigned v = 0;
  if (cudaMemcpyAsync(&v, error_word, sizeof(unsigned), cudaMemcpyDeviceToHost, stream) != cudaSuccess)
    return PKD_ERR_CUDA;
  if (cudaStreamSynchronize(stream) != cudaSuccess) return PKD_ERR_CUDA;
  *host_bits = v;
  if (clear) {
    if (cudaMemsetAsync(error_word, 0, sizeof(int), stream) != cudaSuccess) return PKD_ERR_CUDA;
    if (cudaStreamSynchronize(stream) != cudaSuccess) return PKD_ERR_CUDA;
  }
  return v == 0 ? PKD_OK : PKD_ERR_DEVICE;
}

}  // extern "C"
