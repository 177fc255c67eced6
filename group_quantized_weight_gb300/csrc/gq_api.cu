// C ABI of libgq: argument validation, the launch plan (path choice, split-K), scratch
// management and the timing harness.  The compute itself lives in the kernel files.
#include <atomic>
#include <mutex>
#include <string.h>
#include <unordered_map>
#include <vector>

#include <cstdio>

#include "gq_internal.h"

namespace gq {

static inline bool aligned16(const void *p) { return ((uintptr_t)p & 15u) == 0; }

// gq_set_split_override: process-wide, read at plan time
static std::atomic<int> g_split_override{0};
int split_override() { return g_split_override.load(std::memory_order_relaxed); }
// gq_set_fault_injection: process-wide
static std::atomic<int> g_fault{GQ_FAULT_NONE};
static inline size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }
static inline int ceil_div(int a, int b) { return (a + b - 1) / b; }

int validate(int M, int K, int N, int G, int prec) {
  if (M < 0 || N < 0 || K <= 0) return GQ_ERR_INVALID_ARG;
  if (prec & ~(GQ_W4 | GQ_ZP | GQ_ACT_F32 | GQ_SC_BF16 | GQ_SC_F32 | GQ_OUT_F32 | GQ_STATIC_W |
               GQ_GATE_UP | GQ_ACT_I8 | GQ_ZP_FLOAT))
    return GQ_ERR_INVALID_ARG;
  if ((prec & GQ_ZP_FLOAT) && (prec & GQ_ZP)) return GQ_ERR_INVALID_ARG;   // one zero-point form
  if ((prec & GQ_ZP_FLOAT) && (!(prec & GQ_W4) || (prec & (GQ_GATE_UP | GQ_ACT_I8))))
    return GQ_ERR_UNSUPPORTED;
  if ((prec & GQ_SC_BF16) && (prec & GQ_SC_F32)) return GQ_ERR_INVALID_ARG;
  if (!(G == 32 || G == 64 || G == 128 || G == 256)) return GQ_ERR_UNSUPPORTED;
  if (K < G || K % G != 0) return GQ_ERR_INVALID_ARG;
  if (N % 8 != 0) return GQ_ERR_INVALID_ARG;
  if (prec & GQ_GATE_UP) {
    // W4: whole 16-column tiles of 8 gate and 8 up columns; W8: whole 64-column blocks of 32
    if (N % ((prec & GQ_W4) ? 16 : 64) != 0) return GQ_ERR_INVALID_ARG;
  }
  if (prec & GQ_ACT_I8) {                          // W8A8: INT8 codes, fp32 scales
    if (prec & (GQ_W4 | GQ_ZP | GQ_ACT_F32 | GQ_GATE_UP)) return GQ_ERR_UNSUPPORTED;
    if (!(prec & GQ_SC_F32)) return GQ_ERR_UNSUPPORTED;
    if (K % kChunkK8 != 0) return GQ_ERR_UNSUPPORTED;
    return GQ_OK;
  }
  if (prec & GQ_W4) {
    if (K % kChunkK != 0) return GQ_ERR_UNSUPPORTED;
    if (prec & GQ_ACT_F32) return GQ_ERR_UNSUPPORTED;
  } else {
    if (prec & GQ_ZP) return GQ_ERR_INVALID_ARG;      // INT8 codes are symmetric
    if (K % kChunkK8 != 0) return GQ_ERR_UNSUPPORTED;
    if (!(prec & GQ_ACT_F32)) return GQ_ERR_UNSUPPORTED;
    if (!(prec & GQ_SC_F32)) return GQ_ERR_UNSUPPORTED;
  }
  return GQ_OK;
}

size_t packed_bytes(int K, int N, int prec) {
  if (prec & GQ_W4) return (size_t)ceil_div(N, kTileN) * kTileN * (size_t)K / 2;
  return (size_t)K * N;
}

// device ordinals with a cached SM count and shared-memory limits (others query each time)
constexpr int kMaxDevices = 64;
// SM counts, one per device ordinal, read from the driver once
static std::atomic<int> g_sm_count[kMaxDevices];

int device_sm_count(int *sms) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) { cudaGetLastError(); return GQ_ERR_NO_DEVICE; }
  if (dev >= 0 && dev < kMaxDevices) {
    const int c = g_sm_count[dev].load(std::memory_order_relaxed);
    if (c > 0) {
      *sms = c;
      return GQ_OK;
    }
  }
  if (cudaDeviceGetAttribute(sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
    cudaGetLastError();
    return GQ_ERR_NO_DEVICE;
  }
  if (dev >= 0 && dev < kMaxDevices) g_sm_count[dev].store(*sms, std::memory_order_relaxed);
  return GQ_OK;
}

// the dynamic shared-memory limits this process has set, per (device, kernel)
static std::mutex g_smem_mu;
static std::unordered_map<const void *, size_t> g_smem_set[kMaxDevices];

cudaError_t ensure_dynamic_smem(const void *func, size_t bytes) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const bool cacheable = dev >= 0 && dev < kMaxDevices;
  if (cacheable) {
    std::lock_guard<std::mutex> lk(g_smem_mu);
    auto it = g_smem_set[dev].find(func);
    if (it != g_smem_set[dev].end() && it->second >= bytes) return cudaSuccess;
  }
  e = cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
  if (e == cudaSuccess && cacheable) {
    std::lock_guard<std::mutex> lk(g_smem_mu);
    size_t &v = g_smem_set[dev][func];
    if (v < bytes) v = bytes;
  }
  return e;
}

// Split K into nsplit slices of whole units so that the grid holds about `target` CTAs,
// without exceeding the unit count, a shared-memory budget per CTA and a partial-sum cap.
static int choose_nsplit(int base_ctas, int units, int unit_k, int target,
                         size_t smem_per_k, size_t smem_cap, size_t part_per_split,
                         size_t part_cap) {
  int ns = ceil_div(target, base_ctas);
  if (ns < 1) ns = 1;
  if (ns > units) ns = units;
  while (ns > 1 && (size_t)ns * part_per_split > part_cap) --ns;
  // the widest slice must fit the shared-memory budget
  while (ns < units && (size_t)ceil_div(units, ns) * unit_k * smem_per_k > smem_cap) ++ns;
  return ns;
}

// INT8 codes, N a multiple of 64, few rows: the warp-specialized decode kernel, one CTA per
// SM (a producer warp streaming 2 KB slots for sixteen consumer warps) over a contiguous range
// of (64-column block, group) units; whole blocks per CTA when that keeps the SMs within 10%
// of even, else equal unit ranges with a cross-CTA reduction.  Not a K split: the split
// override leaves it alone.  False (p untouched) when the kernel does not take the shape.
static bool plan_q8_gemv(int Mc, int K, int Nc, int G, int prec, int sms, size_t smem_cap,
                         Plan *p) {
  if (!q8_gemv_supported(Mc, K, Nc, G, prec)) return false;
  const int NB = Nc / 64, gpb = K / G;
  if ((size_t)NB * sizeof(unsigned) > kCounterRegionBytes) return false;
  const int units = NB * gpb, per = ceil_div(NB, sms);
  int grid, split_count, split_mult;
  if (NB >= sms && (double)NB >= 0.9 * (double)sms * per) {
    grid = sms;
    split_count = NB;
    split_mult = gpb;
  } else {
    // equal unit ranges: at least two units per consumer warp, at most one CTA per SM
    grid = ceil_div(units, 32);
    if (grid > sms) grid = sms;
    split_count = units;
    split_mult = 1;
  }
  const int max_cta_units = ceil_div(split_count, grid) * split_mult;
  const size_t smem = q8_gemv_smem_bytes(Mc, K, G, prec, max_cta_units);
  if (smem + 256 > smem_cap) return false;           // 256: its static barriers past 1 KB
  p->path = kPathQ8Gemv;
  p->mt = 1;
  p->m_tile = Mc;
  p->n_tile = 64;
  p->unit_k = G;
  p->units = units;
  p->table_bytes = q8_gemv_table_bytes(max_cta_units);
  p->block_threads = q8_gemv_threads();
  p->smem_bytes = smem;
  p->grid_x = grid;
  p->grid_y = p->grid_z = 1;
  p->split_count = split_count;
  p->split_mult = split_mult;
  if (split_mult == 1) {
    p->part_bytes = round_up(q8_gemv_part_bytes(grid), 256);
    p->counter_bytes = kCounterRegionBytes;
  }
  p->workspace_bytes = p->part_bytes + p->counter_bytes;
  p->nsplit = p->grid_x;
  return true;
}

int make_plan(int M, int K, int N, int G, int prec, int sms, Plan *p) {
  int st = validate(M, K, N, G, prec);
  if (st != GQ_OK) return st;
  if (sms <= 0) return GQ_ERR_INVALID_ARG;
  memset(p, 0, sizeof(*p));
  const int target = sms * 8;          // about two waves of four resident CTAs per SM
  const size_t kPartCap = 64u << 20;   // cap of the partial-sum buffer (bytes)
  const size_t kSmemCap = 96u << 10;   // activation slice budget per CTA (bytes)
  const int Mc = M > 0 ? M : 1;
  const int Nc = N > 0 ? N : 8;
  const size_t kCtaSmemCap = 227u * 1024u - 1024u;   // minus the static shared memory
  // float zero points: the small-batch kernel only
  if ((prec & GQ_ZP_FLOAT) && !(Mc <= kBatchMaxM && batch_supported(Mc, K, G, prec)))
    return GQ_ERR_UNSUPPORTED;
  // W8A8 (GQ_ACT_I8), M <= 4: the warp-specialized decode kernel with dp4a group dots (on the
  // Q8_0 shape 8.3 / 8.8 / 10.0 / 10.1 us for one to four rows against 10.5 / 10.9 / 11.6 /
  // 11.7 for the block kernel below)
  if ((prec & GQ_ACT_I8) && plan_q8_gemv(Mc, K, Nc, G, prec, sms, kCtaSmemCap, p)) return GQ_OK;
  // W8A8 (GQ_ACT_I8): integer group dots, 64 columns x one K slice x 32 rows per CTA
  if (prec & GQ_ACT_I8) {
    const int ks = q8a8_slices(Mc, K, Nc, G, sms, kPartCap, split_override());
    if (ks < 1) return GQ_ERR_UNSUPPORTED;
    p->path = kPathQ8A8;
    p->m_tile = Mc < 32 ? Mc : 32;
    p->n_tile = 64;
    p->unit_k = G;
    p->units = K / G;
    p->nsplit = ks;
    p->grid_x = ceil_div(Nc, 64) * ks;
    p->grid_y = 1;
    p->grid_z = ceil_div(Mc, 32);
    p->block_threads = 256;
    p->smem_bytes = q8a8_smem_bytes(Mc, K, G, ks);
    if (ks > 1) {
      p->part_bytes = round_up((size_t)ks * Mc * Nc * sizeof(float), 256);
      p->counter_bytes = kCounterRegionBytes;
      if ((size_t)p->grid_z * ceil_div(Nc, 64) * sizeof(unsigned) > kCounterRegionBytes)
        return GQ_ERR_UNSUPPORTED;
    }
    p->workspace_bytes = p->part_bytes + p->counter_bytes;
    return GQ_OK;
  }
  // warp-specialized decode (M <= 4): one CTA per SM (a producer warp streaming 2 KB slots
  // for sixteen consumer warps that decode them) over a contiguous range of (tile, 256-k slot)
  // pairs; whole tiles per CTA when that keeps the SMs within 10% of even, else equal slot
  // ranges with a cross-CTA reduction.  Shapes whose activations and tables do not fit the
  // shared memory take the striped kernel below.
  if (gemv_supported(Mc, K, G, prec)) {
    const int T = ceil_div(Nc, kTileN), spt = K / stripe_slot_k();
    const int units = T * spt, per = ceil_div(T, sms);
    int grid, split_count, split_mult;
    if (T >= sms && (double)T >= 0.9 * (double)sms * per) {
      grid = sms;
      split_count = T;
      split_mult = spt;
    } else {
      // equal slot ranges: at least two slots per consumer warp, at most one CTA per SM
      grid = ceil_div(units, 32);
      if (grid > sms) grid = sms;
      split_count = units;
      split_mult = 1;
    }
    const int max_cta_slots = ceil_div(split_count, grid) * split_mult;
    const size_t smem = gemv_smem_bytes(Mc, K, G, prec, max_cta_slots);
    if (smem + 256 <= kCtaSmemCap) {                // 256: its static barriers past 1 KB
      p->path = kPathGemv;
      p->mt = 1;
      p->m_tile = 4;
      p->n_tile = kTileN;
      p->unit_k = stripe_slot_k();
      p->units = units;
      p->table_bytes = gemv_table_bytes(G, prec, max_cta_slots);
      p->block_threads = gemv_threads();
      p->smem_bytes = smem;
      p->grid_x = grid;
      p->grid_y = p->grid_z = 1;
      p->split_count = split_count;
      p->split_mult = split_mult;
      if (split_mult == 1) {
        p->part_bytes = round_up((size_t)grid * 2 * 4 * kTileN * sizeof(float), 256);
        p->counter_bytes = kCounterRegionBytes;
        if ((size_t)T * sizeof(unsigned) > kCounterRegionBytes) return GQ_ERR_UNSUPPORTED;
      }
      p->workspace_bytes = p->part_bytes + p->counter_bytes;
      p->nsplit = p->grid_x;
      return GQ_OK;
    }
  }
  // striped persistent decode (M <= 8): one CTA of kStrWarps warps per SM over a
  // contiguous range of (tile, 256-k slot) pairs; whole tiles per CTA when that keeps the
  // SMs within 10% of even, else equal slot ranges with a cross-CTA reduction
  const int slots = stripe_supported(Mc, K, G, prec) && !(prec & GQ_ZP_FLOAT)
                        ? stripe_slots_for(Mc, K, G, prec, kCtaSmemCap)
                        : 0;
  if (slots >= 2) {
    p->path = kPathStripe;
    p->mt = Mc <= 4 ? 1 : 2;   // MMA blocks
    p->m_tile = 8;
    p->n_tile = kTileN;
    p->unit_k = stripe_slot_k();
    const int T = ceil_div(Nc, kTileN), spt = K / p->unit_k;
    p->units = T * spt;
    p->slots = slots;
    p->block_threads = kStrWarps * 32;
    p->smem_bytes = stripe_smem_bytes(Mc, K, G, prec, slots);
    p->grid_y = p->grid_z = 1;
    const int per = ceil_div(T, sms);
    if (T >= sms && (double)T >= 0.9 * (double)sms * per) {
      p->grid_x = sms;
      p->split_count = T;
      p->split_mult = spt;
      p->workspace_bytes = 0;
    } else {
      int grid = ceil_div(p->units, kStrWarps);
      if (grid > sms) grid = sms;
      p->grid_x = grid;
      p->split_count = p->units;
      p->split_mult = 1;
      p->part_bytes = round_up((size_t)grid * 2 * 8 * kTileN * sizeof(float), 256);
      p->counter_bytes = kCounterRegionBytes;
      if ((size_t)T * sizeof(unsigned) > kCounterRegionBytes) return GQ_ERR_UNSUPPORTED;
      p->workspace_bytes = p->part_bytes + p->counter_bytes;
    }
    p->nsplit = p->grid_x;
    return GQ_OK;
  }
  // INT8 codes with fp32 activations, M <= 4: the warp-specialized decode kernel (on the Q8_0
  // shape 9.4 / 10.6 / 13.7 / 13.7 us for one to four rows against 11.5 / 13.3 / 16.7 / 16.9
  // for the block kernel below)
  if (plan_q8_gemv(Mc, K, Nc, G, prec, sms, kCtaSmemCap, p)) return GQ_OK;
  // INT8 codes, 5 <= M <= 32: BF16 tensor cores, 64 columns x one K slice per CTA (up to 4
  // rows the CUDA-core kernel below is faster: it is load-latency-bound there)
  if (Mc > 4 && Mc <= 32 && q8_mma_supported(Mc, K, G, prec) &&
      q8_mma_slices(Mc, K, Nc, G, sms, kPartCap, 0) >= 1) {
    const int ks = q8_mma_slices(Mc, K, Nc, G, sms, kPartCap, split_override());
    if (ks < 1) return GQ_ERR_UNSUPPORTED;   // a forced count this kernel cannot take
    {
      p->path = kPathQ8Mma;
      p->m_tile = (Mc + 7) / 8 * 8;
      p->mt = (Mc + 7) / 8;
      p->n_tile = 64;
      p->unit_k = G;
      p->units = K / G;
      p->nsplit = ks;
      p->grid_x = ceil_div(Nc, 64) * ks;
      p->grid_y = p->grid_z = 1;
      p->block_threads = 256;
      p->smem_bytes = q8_mma_smem_bytes(Mc, K, G, ks);
      if (ks > 1) {
        p->part_bytes = round_up((size_t)ks * Mc * Nc * sizeof(float), 256);
        p->counter_bytes = kCounterRegionBytes;
        if ((size_t)ceil_div(Nc, 64) * sizeof(unsigned) > kCounterRegionBytes)
          return GQ_ERR_UNSUPPORTED;
      }
      p->workspace_bytes = p->part_bytes + p->counter_bytes;
      return GQ_OK;
    }
  }
  // INT8 codes, M <= 32: CUDA-core FP32 kernel, 64 columns x one K slice per CTA
  if (Mc <= kQ8BlockMaxM && q8_block_supported(Mc, K, G, prec) &&
      q8_block_slices(Mc, K, Nc, G, sms, kPartCap, 0) >= 1) {
    const int ks = q8_block_slices(Mc, K, Nc, G, sms, kPartCap, split_override());
    if (ks < 1) return GQ_ERR_UNSUPPORTED;   // a forced count this kernel cannot take
    {
      p->path = kPathQ8Block;
      p->m_tile = Mc;
      p->n_tile = q8_block_cols();
      p->unit_k = G;
      p->units = K / G;
      p->nsplit = ks;
      p->grid_x = ceil_div(Nc, p->n_tile) * ks;
      p->grid_y = p->grid_z = 1;
      p->block_threads = q8_block_threads();
      p->smem_bytes = q8_block_smem_bytes(Mc, K, G, ks);
      if (ks > 1) {
        p->part_bytes = round_up((size_t)ks * Mc * Nc * sizeof(float), 256);
        p->counter_bytes = kCounterRegionBytes;
        if ((size_t)ceil_div(Nc, p->n_tile) * sizeof(unsigned) > kCounterRegionBytes)
          return GQ_ERR_UNSUPPORTED;
      }
      p->workspace_bytes = p->part_bytes + p->counter_bytes;
      return GQ_OK;
    }
  }
  // the fused gate+up epilogue lives in the decode and small-batch kernels only
  const bool gate_up = (prec & GQ_GATE_UP) != 0;
  if (!gate_up && M >= ((prec & GQ_ZP) ? kPrefillMinMZp : kPrefillMinM) &&
      !(prec & GQ_ZP_FLOAT) &&
      prefill_supported(M, K, N, G, prec)) {
    // M >= 25 (33 with zero points): TMA + tcgen05 persistent kernel, one CTA per SM.  Activation tiles of 64,
    // 128 or 256 rows (the MMA's N) so that few rows do not pay for a 256-row product, and
    // the deepest TMA ring that fits.  The kernel can also split K into slices of whole
    // groups (a last-arriver reduction of FP32 partials), but on GB300 every split measured
    // slower than none: a slice's fixed costs (pipeline start, partial sums out and back)
    // are worth more than the SMs the unsplit grid leaves idle, so the split is only taken
    // when a caller forces it
    p->path = kPathPrefill;
    const int BM = M <= 64 ? 64 : M <= 128 ? 128 : 256;
    p->m_tile = BM;
    p->n_tile = 128;
    p->unit_k = G;
    p->units = K / G;
    const int tiles = ceil_div(N, 128) * ceil_div(M, BM);
    int ks = 1;
    if (split_override() != 0) {
      const int fs = split_override() == -1 ? (p->units < 16 ? p->units : 16) : split_override();
      if (fs < 1 || fs > p->units || (fs > 1 && (size_t)fs * M * N * 4 > kPartCap))
        return GQ_ERR_UNSUPPORTED;
      ks = fs;
    }
    p->nsplit = ks;
    p->grid_x = tiles * ks < sms ? tiles * ks : sms;
    p->grid_y = p->grid_z = 1;
    p->block_threads = kPrefillThreads;
    p->slots = prefill_stages(BM, kCtaSmemCap);
    p->smem_bytes = prefill_smem_bytes(BM, p->slots);
    if (ks > 1) {
      p->part_bytes = round_up((size_t)ks * M * N * sizeof(float), 256);
      p->counter_bytes = kCounterRegionBytes;
      if ((size_t)tiles * 8 * sizeof(unsigned) > kCounterRegionBytes) return GQ_ERR_UNSUPPORTED;
    }
    p->workspace_bytes = p->part_bytes + p->counter_bytes;
    return GQ_OK;
  }
  // small batch (M <= 32, or up to 64 with G = 32): persistent CTAs over (K slice, tile
  // range) pairs, activation
  // slices in shared memory, slices added by the last CTA of each tile range
  if (Mc <= kBatchMaxM && batch_supported(Mc, K, G, prec)) {
    int ksl = batch_slice_k(Mc, K);
    const int forced = split_override();
    if (forced != 0 && batch_slots_for(Mc, ksl, G, prec, kCtaSmemCap) >= 2) {
      // a forced slice count: K/forced must be a whole number of 256-k slots
      const int slots_k = K / 256, fs = forced == -1 ? slots_k : forced;
      if (fs < 1 || fs > slots_k || slots_k % fs != 0) return GQ_ERR_UNSUPPORTED;
      ksl = K / fs;
      if (batch_slots_for(Mc, ksl, G, prec, kCtaSmemCap) < 2) return GQ_ERR_UNSUPPORTED;
      if (fs > 1 && (size_t)fs * Mc * Nc * 4 > kPartCap) return GQ_ERR_UNSUPPORTED;
    }
    const int slots = batch_slots_for(Mc, ksl, G, prec, kCtaSmemCap);
    // split K needs one arrival counter per (row block, 16-column tile)
    const bool ctr_ok = K == ksl || (size_t)ceil_div(Mc, 32) * ceil_div(Nc, kTileN) *
                                            sizeof(unsigned) <= kCounterRegionBytes;
    if (slots >= 2 && ctr_ok) {
      const int ks = K / ksl, rb = ceil_div(Mc, 32);
      int cps = sms / (ks * rb);
      if (cps < 1) cps = 1;
      p->path = kPathBatch;
      p->mt = 4;
      p->m_tile = 32;
      p->n_tile = kTileN;
      p->unit_k = ksl;
      p->units = ks;
      p->nsplit = ks;
      p->split_count = cps;
      p->slots = slots;
      p->grid_x = ks * cps;
      p->grid_y = 1;
      p->grid_z = rb;
      p->block_threads = batch_threads(Mc);
      p->smem_bytes = batch_smem_bytes(Mc, ksl, G, prec, slots);
      if (ks > 1) {
        p->part_bytes = round_up((size_t)ks * Mc * Nc * sizeof(float), 256);
        p->counter_bytes = kCounterRegionBytes;
      }
      p->workspace_bytes = p->part_bytes + p->counter_bytes;
      return GQ_OK;
    }
  }
  if (prec & (GQ_ZP_FLOAT | GQ_GATE_UP)) return GQ_ERR_UNSUPPORTED;
  if (prec & GQ_W4) {
    p->path = kPathMmaDecode;
    const int rows = Mc < 8 * kDecMaxMT ? Mc : 8 * kDecMaxMT;
    p->mt = ceil_div(rows, 8);
    p->m_tile = 8 * p->mt;
    p->n_tile = kDecWarps * kTileN;
    p->unit_k = G > kChunkK ? G : kChunkK;
    p->units = K / p->unit_k;
    p->grid_x = ceil_div(Nc, p->n_tile);
    p->grid_z = ceil_div(Mc, p->m_tile);
    p->block_threads = kDecWarps * 32;
    const int rows_staged = Mc < p->m_tile ? Mc : p->m_tile;
    p->nsplit = choose_nsplit(p->grid_x * p->grid_z, p->units, p->unit_k, target,
                              (size_t)rows_staged * 2, kSmemCap, (size_t)Mc * Nc * 4, kPartCap);
    if (split_override() != 0) {
      const int fs = split_override() == -1 ? p->units : split_override();
      if (fs < 1 || fs > p->units || (size_t)fs * Mc * Nc * 4 > kPartCap ||
          (size_t)ceil_div(p->units, fs) * p->unit_k * rows_staged * 2 > kSmemCap)
        return GQ_ERR_UNSUPPORTED;
      p->nsplit = fs;
    }
    const int widest = ceil_div(p->units, p->nsplit) * p->unit_k;
    p->smem_bytes = (size_t)rows_staged * (widest / kChunkK * 32 + 16) * 4;
  } else {
    p->path = kPathQ8Decode;
    int mr = 1;
    while (mr < Mc && mr < kQ8MaxRows) mr *= 2;
    p->m_tile = mr;
    p->n_tile = kQ8Threads;
    p->unit_k = G;
    p->units = K / G;
    p->grid_x = ceil_div(Nc, p->n_tile);
    p->grid_z = ceil_div(Mc, p->m_tile);
    p->block_threads = kQ8Threads;
    const int rows_staged = Mc < p->m_tile ? Mc : p->m_tile;
    // partial sums may cost at most a quarter of the weight bytes (or one output's worth)
    size_t cap = (size_t)K * Nc / 4;
    if (cap < (size_t)Mc * Nc * 4) cap = (size_t)Mc * Nc * 4;
    if (cap > kPartCap) cap = kPartCap;
    p->nsplit = choose_nsplit(p->grid_x * p->grid_z, p->units, p->unit_k, target,
                              (size_t)rows_staged * 4, kSmemCap, (size_t)Mc * Nc * 4, cap);
    if (split_override() != 0) {
      const int fs = split_override() == -1 ? p->units : split_override();
      if (fs < 1 || fs > p->units || (size_t)fs * Mc * Nc * 4 > kPartCap ||
          (size_t)ceil_div(p->units, fs) * p->unit_k * rows_staged * 4 > kSmemCap)
        return GQ_ERR_UNSUPPORTED;
      p->nsplit = fs;
    }
    const int widest = ceil_div(p->units, p->nsplit) * p->unit_k;
    p->smem_bytes = (size_t)rows_staged * widest * 4;
  }
  if (p->smem_bytes > (200u << 10)) return GQ_ERR_UNSUPPORTED;
  p->grid_y = p->nsplit;
  if (p->nsplit > 1) {
    p->part_bytes = round_up((size_t)p->nsplit * Mc * Nc * sizeof(float), 256);
    p->counter_bytes = kCounterRegionBytes;
    if ((size_t)p->grid_x * p->grid_z * sizeof(unsigned) > kCounterRegionBytes)
      return GQ_ERR_UNSUPPORTED;
  }
  p->workspace_bytes = p->part_bytes + p->counter_bytes;
  return GQ_OK;
}

// Bytes of arrival counters the kernels of plan p index (a prefix of the counter region);
// 0 when the plan uses none.
size_t plan_counter_bytes_used(const Plan &p, int M, int N) {
  if (p.counter_bytes == 0) return 0;
  const int Nc = N > 0 ? N : 8;
  size_t n = 0;
  switch (p.path) {
    case kPathQ8A8: n = (size_t)p.grid_z * ceil_div(Nc, 64); break;
    case kPathStripe:
    case kPathGemv: n = (size_t)ceil_div(Nc, kTileN); break;
    case kPathPrefill: n = (size_t)ceil_div(Nc, 128) * ceil_div(M > 0 ? M : 1, p.m_tile) * 8; break;
    case kPathQ8Mma: n = (size_t)ceil_div(Nc, 64); break;
    case kPathQ8Block: n = (size_t)ceil_div(Nc, p.n_tile); break;
    case kPathQ8Gemv: n = (size_t)ceil_div(Nc, 64); break;
    case kPathBatch: n = (size_t)p.grid_z * ceil_div(Nc, kTileN); break;
    default: n = (size_t)p.grid_x * p.grid_z; break;
  }
  const size_t b = round_up(n * sizeof(unsigned), 16);
  return b < p.counter_bytes ? b : p.counter_bytes;
}

// ------------------------------------------------------------------ scratch per device

struct DevScratch {
  void *ptr = nullptr;
  size_t bytes = 0;
  bool user = false;
};
static std::mutex g_mu;
static std::vector<DevScratch> g_scratch;

static int get_scratch(size_t need, void **out) {
  *out = nullptr;
  if (need == 0) return GQ_OK;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) { cudaGetLastError(); return GQ_ERR_NO_DEVICE; }
  std::lock_guard<std::mutex> lk(g_mu);
  if ((int)g_scratch.size() <= dev) g_scratch.resize(dev + 1);
  DevScratch &d = g_scratch[dev];
  if (d.user) {
    if (d.bytes < need) return GQ_ERR_WORKSPACE;
    *out = d.ptr;
    return GQ_OK;
  }
  if (g_fault.load(std::memory_order_relaxed) == GQ_FAULT_WORKSPACE) {
    note_cuda_error_code("workspace allocation (injected)", 0);
    return GQ_ERR_CUDA;
  }
  if (d.bytes < need) {
    if (d.ptr) {
      if (cudaDeviceSynchronize() != cudaSuccess || cudaFree(d.ptr) != cudaSuccess) {
        cudaGetLastError();
        return GQ_ERR_CUDA;
      }
      d.ptr = nullptr;
      d.bytes = 0;
    }
    size_t sz = round_up(need, 1u << 20);
    void *p = nullptr;
    if (cudaMalloc(&p, sz) != cudaSuccess) { cudaGetLastError(); return GQ_ERR_CUDA; }
    if (cudaMemset(p, 0, sz) != cudaSuccess || cudaDeviceSynchronize() != cudaSuccess) {
      cudaGetLastError();
      cudaFree(p);
      return GQ_ERR_CUDA;
    }
    d.ptr = p;
    d.bytes = sz;
  }
  *out = d.ptr;
  return GQ_OK;
}

cudaError_t launch_plan(const Plan &p, int M, int K, int N, int G, int prec, const void *A,
                        const void *Wq, const void *scales, const void *zeros, void *out,
                        float *part, unsigned *counters, cudaStream_t s) {
  switch (p.path) {
    case kPathPrefill:
      return launch_prefill(p, M, K, N, G, prec, A, Wq, scales, zeros, out, part, counters, s);
    case kPathGemv:
      return launch_gemv(p, M, K, N, G, prec, A, Wq, scales, zeros, out, part, counters, s);
    case kPathStripe:
      return launch_stripe_decode(p, M, K, N, G, prec, A, Wq, scales, zeros, out, part,
                                  counters, s);
    case kPathBatch:
      return launch_batch(p, M, K, N, G, prec, A, Wq, scales, zeros, out, part, counters, s);
    case kPathMmaDecode:
      return launch_mma_decode(p, M, K, N, G, prec, A, Wq, scales, zeros, out, part, counters,
                               s);
    case kPathQ8Mma:
      return launch_q8_mma(p, M, K, N, G, prec, A, Wq, scales, out, part, counters, s);
    case kPathQ8Block:
      return launch_q8_block(p, M, K, N, G, prec, A, Wq, scales, out, part, counters, s);
    case kPathQ8Gemv:
      return launch_q8_gemv(p, M, K, N, G, prec, A, nullptr, Wq, scales, out, part, counters,
                            s);
    case kPathQ8Decode:
      return launch_q8_decode(p, M, K, N, G, prec, A, Wq, scales, out, part, counters, s);
    default:
      return cudaErrorInvalidValue;
  }
}

// true (and the detail noted) when gq_set_fault_injection asked launches to fail
bool launch_fault_injected() {
  if (g_fault.load(std::memory_order_relaxed) != GQ_FAULT_LAUNCH) return false;
  note_cuda_error_code("launch (injected)", 0);
  return true;
}

static thread_local char g_detail[160];
void note_cuda_error(const char *where, cudaError_t e) {
  snprintf(g_detail, sizeof(g_detail), "%s: %s", where, cudaGetErrorName(e));
}
void note_cuda_error_code(const char *where, int code) {
  snprintf(g_detail, sizeof(g_detail), "%s: error %d", where, code);
}

}  // namespace gq

using namespace gq;

extern "C" {

const char *gq_last_error_detail(void) { return gq::g_detail; }

const char *gq_status_string(int status) {
  switch (status) {
    case GQ_OK: return "ok";
    case GQ_ERR_INVALID_ARG: return "invalid argument";
    case GQ_ERR_UNSUPPORTED: return "unsupported shape or operand combination";
    case GQ_ERR_ALIGNMENT: return "pointer not 16-byte aligned";
    case GQ_ERR_WORKSPACE: return "workspace too small";
    case GQ_ERR_CUDA: return "CUDA error";
    case GQ_ERR_TIMEOUT: return "device-side wait timed out";
    case GQ_ERR_NO_DEVICE: return "no usable CUDA device";
    default: return "unknown status";
  }
}

int gq_set_wait_limit(long long cycles) {
  if (cycles != 0 && (cycles < 10000ll || cycles > 100000000000ll)) return GQ_ERR_INVALID_ARG;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) { cudaGetLastError(); return GQ_ERR_NO_DEVICE; }
  const long long v = cycles == 0 ? 4000000000ll : cycles;
  const int r = gemv_set_wait_limit(v) | stripe_set_wait_limit(v) | batch_set_wait_limit(v) |
                prefill_set_wait_limit(v) | fp8_set_wait_limit(v) | q8_gemv_set_wait_limit(v);
  if (r != 0) {
    note_cuda_error_code("gq_set_wait_limit", r);
    cudaGetLastError();
    return GQ_ERR_CUDA;
  }
  return GQ_OK;
}

int gq_set_fault_injection(int fault) {
  if (fault < GQ_FAULT_NONE || fault > GQ_FAULT_DEVICE_WAIT) return -1;
  const int prev = g_fault.load();
  // the device-side form is a launch parameter of the warp-specialized decode kernel
  gemv_set_withhold(fault == GQ_FAULT_DEVICE_WAIT);
  g_fault.store(fault);
  return prev;
}

int gq_set_split_override(int n) {
  if (n < -1) return -2;
  return g_split_override.exchange(n);
}

int gq_zsplit(int units, int nsplit, int z, int *begin, int *end) {
  if (!begin || !end || units < 0 || nsplit < 1 || z < 0 || z >= nsplit) return GQ_ERR_INVALID_ARG;
  const int base = units / nsplit, rem = units % nsplit;
  *begin = z * base + (z < rem ? z : rem);
  *end = *begin + base + (z < rem ? 1 : 0);
  return GQ_OK;
}

int gq_packed_bytes(int K, int N, int G, int prec, size_t *bytes) {
  if (!bytes) return GQ_ERR_INVALID_ARG;
  int st = validate(1, K, N, G, prec);
  if (st != GQ_OK) return st;
  *bytes = packed_bytes(K, N, prec);
  return GQ_OK;
}

int gq_plan(int M, int K, int N, int G, int prec, int sm_count, gq_plan_t *plan) {
  if (!plan) return GQ_ERR_INVALID_ARG;
  int sms = sm_count;
  if (sms <= 0) {
    int st = device_sm_count(&sms);
    if (st != GQ_OK) return st;
  }
  Plan p;
  int st = make_plan(M, K, N, G, prec, sms, &p);
  if (st != GQ_OK) return st;
  plan->path = p.path;
  plan->nsplit = p.nsplit;
  plan->m_tile = p.m_tile;
  plan->n_tile = p.n_tile;
  plan->grid_x = p.grid_x;
  plan->grid_y = p.grid_y;
  plan->grid_z = p.grid_z;
  plan->block_threads = p.block_threads;
  plan->smem_bytes = p.smem_bytes;
  plan->workspace_bytes = p.workspace_bytes;
  return GQ_OK;
}

int gq_workspace_size(int M, int K, int N, int G, int prec, size_t *bytes) {
  if (!bytes) return GQ_ERR_INVALID_ARG;
  int sms = 0;
  int st = device_sm_count(&sms);
  if (st != GQ_OK) return st;
  Plan p;
  st = make_plan(M, K, N, G, prec, sms, &p);
  if (st != GQ_OK) return st;
  *bytes = (M == 0 || N == 0) ? 0 : p.workspace_bytes;
  return GQ_OK;
}

int gq_set_workspace(void *dev_ptr, size_t bytes) {
  if (((uintptr_t)dev_ptr & 255u) != 0) return GQ_ERR_ALIGNMENT;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) { cudaGetLastError(); return GQ_ERR_NO_DEVICE; }
  std::lock_guard<std::mutex> lk(g_mu);
  if ((int)g_scratch.size() <= dev) g_scratch.resize(dev + 1);
  DevScratch &d = g_scratch[dev];
  if (!d.user && d.ptr) {
    if (cudaDeviceSynchronize() != cudaSuccess) { cudaGetLastError(); return GQ_ERR_CUDA; }
    cudaFree(d.ptr);
  }
  d.ptr = nullptr;
  d.bytes = 0;
  d.user = false;
  if (dev_ptr && bytes) {
    if (cudaMemset(dev_ptr, 0, bytes) != cudaSuccess || cudaDeviceSynchronize() != cudaSuccess) {
      cudaGetLastError();
      return GQ_ERR_CUDA;
    }
    d.ptr = dev_ptr;
    d.bytes = bytes;
    d.user = true;
  }
  return GQ_OK;
}

int gq_pack_weights(int K, int N, int G, int prec, const void *codes, void *packed,
                    void *stream) {
  int st = validate(1, K, N, G, prec);
  if (st != GQ_OK) return st;
  if (N == 0) return GQ_OK;
  if (!codes || !packed) return GQ_ERR_INVALID_ARG;
  if (!aligned16(codes) || !aligned16(packed)) return GQ_ERR_ALIGNMENT;
  cudaStream_t s = (cudaStream_t)stream;
  cudaError_t e;
  if (prec & GQ_W4)
    e = launch_pack_w4(K, N, (const uint32_t *)codes, (uint32_t *)packed,
                       (prec & GQ_GATE_UP) != 0, s);
  else
    e = launch_pack_w8(K, N, (const int8_t *)codes, (uint8_t *)packed,
                       (prec & GQ_GATE_UP) != 0, s);
  return e == cudaSuccess ? GQ_OK : GQ_ERR_CUDA;
}

static int gemm_a8_impl(int M, int K, int N, int G, int prec, const void *Aq,
                        const void *a_scales, const void *Wq, const void *scales, void *out,
                        void *stream);

}  // extern "C"

// Everything gq_gemm checks and prepares before its launch: the arguments, the plan and the
// scratch.  *empty is set when there is nothing to compute (M or N is 0).
static int gemm_prepare(int M, int K, int N, int G, int prec, const void *A, const void *Wq,
                        const void *scales, const void *zeros, const void *out, Plan *p,
                        void **ws, bool *empty) {
  *empty = false;
  if (prec & GQ_ACT_I8) return GQ_ERR_INVALID_ARG;   // needs the activation scales: gq_gemm_a8
  int st = validate(M, K, N, G, prec);
  if (st != GQ_OK) return st;
  if (M == 0 || N == 0) {
    *empty = true;
    return GQ_OK;
  }
  if (!A || !Wq || !scales || !out) return GQ_ERR_INVALID_ARG;
  if (((prec & (GQ_ZP | GQ_ZP_FLOAT)) != 0) != (zeros != nullptr)) return GQ_ERR_INVALID_ARG;
  if (!aligned16(A) || !aligned16(Wq) || !aligned16(scales) || !aligned16(out) ||
      (zeros && !aligned16(zeros)))
    return GQ_ERR_ALIGNMENT;
  int sms = 0;
  st = device_sm_count(&sms);
  if (st != GQ_OK) return st;
  st = make_plan(M, K, N, G, prec, sms, p);
  if (st != GQ_OK) return st;
  return get_scratch(p->workspace_bytes, ws);
}

static int gemm_launch(const Plan &p, int M, int K, int N, int G, int prec, const void *A,
                       const void *Wq, const void *scales, const void *zeros, void *out,
                       void *ws, cudaStream_t s) {
  unsigned *counters = (unsigned *)ws;
  float *part = ws ? (float *)((char *)ws + p.counter_bytes) : nullptr;
  if (launch_fault_injected()) return GQ_ERR_CUDA;
  const cudaError_t e = launch_plan(p, M, K, N, G, prec, A, Wq, scales, zeros, out, part,
                                    counters, s);
  if (e != cudaSuccess) {
    note_cuda_error("launch", e);
    cudaGetLastError();
    return GQ_ERR_CUDA;
  }
  return GQ_OK;
}

int gq::gemm_impl(int M, int K, int N, int G, int prec, const void *A, const void *Wq,
                  const void *scales, const void *zeros, void *out, void *stream) {
  Plan p;
  void *ws = nullptr;
  bool empty = false;
  const int st = gemm_prepare(M, K, N, G, prec, A, Wq, scales, zeros, out, &p, &ws, &empty);
  if (st != GQ_OK || empty) return st;
  return gemm_launch(p, M, K, N, G, prec, A, Wq, scales, zeros, out, ws, (cudaStream_t)stream);
}

extern "C" {

int gq_gemm(int M, int K, int N, int G, int prec, const void *A, const void *Wq,
            const void *scales, const void *zeros, void *out, void *stream) {
  return gemm_impl(M, K, N, G, prec, A, Wq, scales, zeros, out, stream);
}

int gq_gemm_host(int M, int K, int N, int G, int prec, const void *A_host, void *A_dev,
                 const void *Wq, const void *scales, const void *zeros, void *out_dev,
                 void *out_host, void *stream) {
  int st = validate(M, K, N, G, prec);
  if (st != GQ_OK) return st;
  if (M == 0 || N == 0) return GQ_OK;
  if (!A_host || !out_host) return GQ_ERR_INVALID_ARG;
  Plan p;
  void *ws = nullptr;
  bool empty = false;
  st = gemm_prepare(M, K, N, G, prec, A_dev, Wq, scales, zeros, out_dev, &p, &ws, &empty);
  if (st != GQ_OK || empty) return st;
  const size_t a_bytes = (size_t)M * K * ((prec & GQ_ACT_F32) ? 4 : 2);
  const size_t o_cols = (prec & GQ_GATE_UP) ? (size_t)N / 2 : (size_t)N;
  const size_t o_bytes = (size_t)M * o_cols * ((prec & GQ_OUT_F32) ? 4 : 2);
  const cudaStream_t s = (cudaStream_t)stream;
  cudaError_t e = cudaMemcpyAsync(A_dev, A_host, a_bytes, cudaMemcpyHostToDevice, s);
  if (e != cudaSuccess) {
    note_cuda_error("cudaMemcpyAsync(activations to the device)", e);
    cudaGetLastError();
    return GQ_ERR_CUDA;
  }
  st = gemm_launch(p, M, K, N, G, prec, A_dev, Wq, scales, zeros, out_dev, ws, s);
  if (st != GQ_OK) return st;
  e = cudaMemcpyAsync(out_host, out_dev, o_bytes, cudaMemcpyDeviceToHost, s);
  if (e != cudaSuccess) {
    note_cuda_error("cudaMemcpyAsync(output to the host)", e);
    cudaGetLastError();
    return GQ_ERR_CUDA;
  }
  return GQ_OK;
}

static int gemm_a8_impl(int M, int K, int N, int G, int prec, const void *Aq,
                        const void *a_scales, const void *Wq, const void *scales, void *out,
                        void *stream) {
  if (!(prec & GQ_ACT_I8)) return GQ_ERR_INVALID_ARG;
  int st = validate(M, K, N, G, prec);
  if (st != GQ_OK) return st;
  if (M == 0 || N == 0) return GQ_OK;
  if (!Aq || !a_scales || !Wq || !scales || !out) return GQ_ERR_INVALID_ARG;
  if (!aligned16(Aq) || !aligned16(a_scales) || !aligned16(Wq) || !aligned16(scales) ||
      !aligned16(out))
    return GQ_ERR_ALIGNMENT;
  int sms = 0;
  st = device_sm_count(&sms);
  if (st != GQ_OK) return st;
  Plan p;
  st = make_plan(M, K, N, G, prec, sms, &p);
  if (st != GQ_OK) return st;
  void *ws = nullptr;
  st = get_scratch(p.workspace_bytes, &ws);
  if (st != GQ_OK) return st;
  unsigned *counters = (unsigned *)ws;
  float *part = ws ? (float *)((char *)ws + p.counter_bytes) : nullptr;
  if (launch_fault_injected()) return GQ_ERR_CUDA;
  const cudaError_t e =
      p.path == kPathQ8Gemv
          ? launch_q8_gemv(p, M, K, N, G, prec, Aq, (const float *)a_scales, Wq, scales, out,
                           part, counters, (cudaStream_t)stream)
          : launch_q8a8(p, M, K, N, G, prec, (const int8_t *)Aq, (const float *)a_scales, Wq,
                        scales, out, part, counters, (cudaStream_t)stream);
  if (e != cudaSuccess) {
    note_cuda_error("launch", e);
    cudaGetLastError();
    return GQ_ERR_CUDA;
  }
  return GQ_OK;
}

int gq_gemm_a8(int M, int K, int N, int G, int prec, const void *Aq, const void *a_scales,
               const void *Wq, const void *scales, void *out, void *stream) {
  return gemm_a8_impl(M, K, N, G, prec, Aq, a_scales, Wq, scales, out, stream);
}

int gq_quantize_act(int M, int K, int G, int prec, const void *A, void *Aq, void *a_scales,
                    void *stream) {
  if (prec & ~GQ_ACT_F32) return GQ_ERR_INVALID_ARG;
  if (M < 0 || K <= 0) return GQ_ERR_INVALID_ARG;
  if (!(G == 32 || G == 64 || G == 128 || G == 256) || K % G != 0 || K % 16 != 0)
    return GQ_ERR_INVALID_ARG;
  if (M == 0) return GQ_OK;
  if (!A || !Aq || !a_scales) return GQ_ERR_INVALID_ARG;
  if (!aligned16(A) || !aligned16(Aq) || !aligned16(a_scales)) return GQ_ERR_ALIGNMENT;
  const cudaError_t e = launch_quantize_act(M, K, G, (prec & GQ_ACT_F32) != 0, A,
                                            (int8_t *)Aq, (float *)a_scales, (cudaStream_t)stream);
  if (e != cudaSuccess) {
    note_cuda_error("launch", e);
    cudaGetLastError();
    return GQ_ERR_CUDA;
  }
  return GQ_OK;
}

int gq_bench_calls(const gq_bench_args *a, gq_bench_result *r) {
  if (!a || !r || a->n_copies < 1 || a->iters < 1 || a->warmup < 0 || !a->Wq || !a->scales)
    return GQ_ERR_INVALID_ARG;
  if ((a->prec & (GQ_ZP | GQ_ZP_FLOAT)) && !a->zeros) return GQ_ERR_INVALID_ARG;
  cudaStream_t s = (cudaStream_t)a->stream;
  if ((a->prec & GQ_ACT_I8) && !a->a_scales) return GQ_ERR_INVALID_ARG;
  auto call = [&](int i) {
    const int c = i % a->n_copies;
    if (a->prec & GQ_ACT_I8)
      return gemm_a8_impl(a->M, a->K, a->N, a->G, a->prec, a->A, a->a_scales, a->Wq[c],
                          a->scales[c], a->out, a->stream);
    return gemm_impl(a->M, a->K, a->N, a->G, a->prec, a->A, a->Wq[c], a->scales[c],
                     (a->prec & (GQ_ZP | GQ_ZP_FLOAT)) ? a->zeros[c] : nullptr, a->out,
                     a->stream);
  };
  int st = GQ_OK;
  for (int i = 0; i < a->warmup && st == GQ_OK; ++i) st = call(i);
  if (st != GQ_OK) return st;
  if (st == GQ_OK && a->warmup == 0) st = call(0);   // make sure scratch exists
  if (st != GQ_OK) return st;
  cudaEvent_t e0, e1;
  if (cudaEventCreate(&e0) != cudaSuccess || cudaEventCreate(&e1) != cudaSuccess) {
    cudaGetLastError();
    return GQ_ERR_CUDA;
  }
  cudaGraph_t graph = nullptr;
  cudaGraphExec_t exec = nullptr;
  int rc = GQ_OK;
  auto cuda_ok = [&](cudaError_t e, const char *where) {
    if (e == cudaSuccess) return true;
    note_cuda_error(where, e);
    rc = GQ_ERR_CUDA;
    return false;
  };
  if (a->use_graph) {
    // capture needs a stream other than the legacy default stream
    if (cuda_ok(cudaStreamBeginCapture(s, cudaStreamCaptureModeThreadLocal), "cudaStreamBeginCapture")) {
      for (int i = 0; i < a->iters && rc == GQ_OK; ++i) rc = call(i);
      cudaGraph_t g2 = nullptr;
      const cudaError_t ee = cudaStreamEndCapture(s, &g2);
      if (rc == GQ_OK) cuda_ok(ee, "cudaStreamEndCapture");
      graph = g2;
    }
    if (rc == GQ_OK) cuda_ok(cudaGraphInstantiate(&exec, graph, 0), "cudaGraphInstantiate");
    if (rc == GQ_OK) cuda_ok(cudaGraphLaunch(exec, s), "cudaGraphLaunch");   // warm
  }
  if (rc == GQ_OK) {
    cudaEventRecord(e0, s);
    if (a->use_graph) {
      cuda_ok(cudaGraphLaunch(exec, s), "cudaGraphLaunch");
    } else {
      for (int i = 0; i < a->iters && rc == GQ_OK; ++i) rc = call(i);
    }
    cudaEventRecord(e1, s);
  }
  {
    const cudaError_t es = cudaStreamSynchronize(s);
    if (rc == GQ_OK) cuda_ok(es, "cudaStreamSynchronize");
  }
  float ms = 0.f;
  if (rc == GQ_OK) cuda_ok(cudaEventElapsedTime(&ms, e0, e1), "cudaEventElapsedTime");
  if (exec) cudaGraphExecDestroy(exec);
  if (graph) cudaGraphDestroy(graph);
  cudaEventDestroy(e0);
  cudaEventDestroy(e1);
  if (rc != GQ_OK) { cudaGetLastError(); return rc; }
  r->us_per_call = 1000.0 * ms / a->iters;
  r->launches_per_call = 1;
  return GQ_OK;
}

int gq_device_error(int clear) {
  const int v = prefill_read_error(clear);
  const int w = stripe_read_error(clear);
  const int x = batch_read_error(clear);
  const int y = fp8_read_error(clear);
  const int g = gemv_read_error(clear);
  const int q = q8_gemv_read_error(clear);
  return v != 0 ? v : (w != 0 ? w : (x != 0 ? x : (y != 0 ? y : (g != 0 ? g : q))));
}

int gq_quantize_act_fp8(int M, int K, int prec, const void *A, void *Aq, void *a_scales,
                        void *stream) {
  if (prec & ~GQ_ACT_F32) return GQ_ERR_INVALID_ARG;
  if (M < 0 || K < 128 || K % 128 != 0) return GQ_ERR_INVALID_ARG;
  if (M == 0) return GQ_OK;
  if (!A || !Aq || !a_scales) return GQ_ERR_INVALID_ARG;
  if (!aligned16(A) || !aligned16(Aq) || !aligned16(a_scales)) return GQ_ERR_ALIGNMENT;
  return launch_quantize_fp8(M, K, (prec & GQ_ACT_F32) != 0, A, Aq, a_scales,
                             (cudaStream_t)stream);
}

int gq_gemm_fp8_block(int M, int K, int N, int prec, const void *A, const void *a_scales,
                      const void *W, const void *w_scales, void *out, void *stream) {
  if (prec & ~GQ_OUT_F32) return GQ_ERR_INVALID_ARG;
  if (M < 0 || N < 0 || K < 128 || K % 128 != 0 || N % 16 != 0) return GQ_ERR_INVALID_ARG;
  if (M == 0 || N == 0) return GQ_OK;
  if (!A || !a_scales || !W || !w_scales || !out) return GQ_ERR_INVALID_ARG;
  if (!aligned16(A) || !aligned16(a_scales) || !aligned16(W) || !aligned16(w_scales) ||
      !aligned16(out))
    return GQ_ERR_ALIGNMENT;
  int sms = 0;
  int st = device_sm_count(&sms);
  if (st != GQ_OK) return st;
  int grid = 0;
  fp8_block_plan(M, N, sms, &grid);
  return launch_fp8_block(M, K, N, prec, A, a_scales, W, w_scales, out, grid,
                          (cudaStream_t)stream);
}

}  // extern "C"
