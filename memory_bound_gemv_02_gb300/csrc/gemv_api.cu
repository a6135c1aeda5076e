// Host side of the GEMV library: argument checks, the launch planner, the
// per-key configuration cache, split-K workspaces and the launches.
//
// The hot call (a cached key) is: validation (pure arithmetic), one
// cudaGetDevice, one hash lookup under a mutex, and one or two kernel
// launches.  Everything that costs more -- device attribute queries,
// cudaFuncSetAttribute, workspace allocation -- happens once, when a key or
// a (device, stream) pair is first seen.  This is the GB300 counterpart of
// TileLang Case Studies Case B.4 / Case E, where per-call kernel building
// cost 11-200 ms against a ~70 us kernel.
#include <cuda_runtime.h>

#include <atomic>
#include <cstdint>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <map>
#include <mutex>
#include <set>
#include <unordered_map>
#include <utility>

#include "gemv.h"
#include "gemv_internal.h"

// Ring waits of the bulk kernel that gave up, on each device that loads this
// library (read and cleared by gemv_wait_timeouts()).
static __device__ uint32_t g_gemv_wait_timeouts;

namespace gemvk {
namespace {

constexpr int64_t kBulkAutoBytes = 768LL << 20;  // the planner's bulk variant: B bytes from which,
constexpr int64_t kBulkAutoMinK = 6144;           // and the row lengths [kBulkAutoMinK, kBulkAutoEndK)
constexpr int64_t kBulkAutoEndK = 8192;           // for which it is chosen
constexpr int64_t kMaxSegment = 32768;  // columns of a staged per CTA (64 KiB of shared memory)
constexpr int kMaxGridSplit = 64;              // most k-segments the planner adds to fill the GPU
constexpr int64_t kMaxSegments = 65536;         // most k-segments of any plan: k <= INT32_MAX in 32768-column segments
constexpr int kAutoVariant = GEMV_VARIANT_TILES;  // the planner's default family
constexpr int kDefaultL2Prefetch = 0;              // tile rounds of L2 prefetch by default
constexpr int kBulkDefaultStages = 2;              // ring buffers per warp of the bulk variant
constexpr int kMaxSmemPerCta = 232448;  // 227 KiB, sm_100-family opt-in limit
constexpr int64_t kSmemPerSm = 233472;  // 228 KiB of shared memory per SM
constexpr int64_t kSmemReservedPerCta = 1024;
constexpr int kMaxDevices = 64;
constexpr int kReduceThreads = 256;

inline int64_t cdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }

// Blocks of the split-K second pass: a thread per row for up to 32
// segments, a warp per row beyond (the kernel's two modes); grid-stride
// loops cover any remainder past the 65535-block cap.
inline unsigned reduce_blocks(int64_t n, int64_t sg) {
  int64_t b = cdiv(n, sg > 32 ? kReduceThreads / 32 : kReduceThreads);
  if (b > 65535) b = 65535;
  return (unsigned)(b < 1 ? 1 : b);
}
inline int64_t round_up(int64_t a, int64_t b) { return cdiv(a, b) * b; }
inline int64_t pow2_ceil(int64_t x) {
  int64_t p = 1;
  while (p < x) p *= 2;
  return p;
}

inline int64_t pow2_floor(int64_t x) {
  int64_t p = 1;
  while (p * 2 <= x) p *= 2;
  return p;
}
inline int out_elem_bytes(int dtype) { return dtype >= 2 ? 4 : 2; }

struct DeviceInfo {
  bool init = false;
  bool ok = false;
  int sm_count = 0;
  int max_smem_optin = 0;
};

struct Key {
  int dev;
  int dtype;
  int aligned;
  int64_t n;
  int64_t k;
  bool operator==(const Key &o) const {
    return dev == o.dev && dtype == o.dtype && aligned == o.aligned && n == o.n && k == o.k;
  }
};

struct KeyHash {
  size_t operator()(const Key &x) const {
    uint64_t h = 1469598103934665603ull;
    auto mix = [&h](uint64_t v) {
      h ^= v;
      h *= 1099511628211ull;
    };
    mix((uint64_t)x.dev);
    mix((uint64_t)x.dtype);
    mix((uint64_t)x.aligned);
    mix((uint64_t)x.n);
    mix((uint64_t)x.k);
    return (size_t)h;
  }
};

struct Workspace {
  float *ptr = nullptr;
  size_t bytes = 0;
};

std::mutex g_mu;
DeviceInfo g_dev[kMaxDevices];
std::unordered_map<Key, gemv_config, KeyHash> g_cache;
std::map<std::pair<int, cudaStream_t>, Workspace> g_ws;
std::set<std::pair<const void *, int>> g_func_attr_set;
std::atomic<int> g_inject{0};
std::atomic<int> g_wait_budget{-1};  // one-shot poll budget of the next bulk launch (-1: none)

uint32_t *g_timeouts_ptr[kMaxDevices] = {};  // device address of g_gemv_wait_timeouts, per device (g_mu)

thread_local gemv_config t_last{};
thread_local bool t_has_last = false;
thread_local int t_cuda_err = 0;

int cuda_fail(cudaError_t e) {
  t_cuda_err = (int)e;
  return GEMV_ERR_CUDA;
}

// Device attributes, queried once per device (caller holds g_mu).
const DeviceInfo &device_info_locked(int dev) {
  DeviceInfo &d = g_dev[dev];
  if (!d.init) {
    d.init = true;
    int major = 0, minor = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) == cudaSuccess &&
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) == cudaSuccess &&
        cudaDeviceGetAttribute(&d.sm_count, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess &&
        cudaDeviceGetAttribute(&d.max_smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) ==
            cudaSuccess) {
      d.ok = (major == 10 && minor == 3);
    }
  }
  return d;
}

// GEMV_LOG=1 in the environment (read once, at the first configuration
// built): one line on stderr for each launch configuration the planner
// builds -- a new key cached by gemv()/gemv_ex()/gemv_fused()/
// gemv_prepare(), or a gemv_plan() call -- giving the key and what it maps
// to.  Off otherwise.
bool log_enabled() {
  static const bool on = [] {
    const char *v = std::getenv("GEMV_LOG");
    return v != nullptr && v[0] == '1' && v[1] == '\0';
  }();
  return on;
}

void log_config(const char *what, int dev, int64_t n, int64_t k, int dtype, bool aligned, const gemv_config &c) {
  if (!log_enabled()) return;
  std::fprintf(stderr,
               "gemv: %s dev=%d n=%lld k=%lld dtype=%d aligned=%d -> variant=%d ctas=%d warps_per_cta=%d "
               "warp_split=%d rows_per_warp=%d unroll=%d grid_split=%d k_segment=%lld stages=%d smem_bytes=%d\n",
               what, dev, (long long)n, (long long)k, dtype, aligned ? 1 : 0, c.variant, c.ctas, c.warps_per_cta,
               c.warp_split, c.rows_per_warp, c.unroll, c.grid_split, (long long)c.k_segment, c.stages, c.smem_bytes);
}

bool valid_W(int W) { return W == 4 || W == 8 || W == 16; }
bool valid_R(int R) { return R == 1 || R == 2 || R == 4; }

bool valid_tiles_RU(int R, int U) {
  return (R == 1 && (U == 8 || U == 4)) || (R == 2 && U == 4) || (R == 4 && U == 2);
}

// Warps per row (S) of the tiles kernel for rows of nt 16-byte blocks: the
// smallest power-of-two split whose slices are at most 1024 blocks (16 KB
// per warp and row; longer slices measured 4-10 % slower at k = 16384) plus
// the at most 32 blocks the kernel folds into a slice's last step (so the
// extra edge block of an unaligned row does not double S: 7168 x 16384 at
// an odd element offset 38.1 us with S = 4, slices of 513 blocks) and that
// gives at least 80 % of the resident warps (sm x 32) a slice, without
// cutting slices below 128 blocks.  Measured on GB300 against every (W, S,
// R) over the workload shapes: this choice is the fastest or within 3 % of
// it.
//
// With split-K (Sg k-segments) every segment of a row is a unit of its own,
// so the fill counts n * S * Sg.  Few rows per CTA can leave most warps of
// the last round of row tiles idle: while a round is less than 75 % full, S
// keeps doubling as long as that fills the rounds better (300 x 100003: 4
// warps per row 21.0 us, 16 warps per row 18.8 us).
int tiles_split(int64_t n, int64_t nt, int W, int sm, int64_t Sg, int NCLS, int cps_warps) {
  int S = (int)pow2_ceil(cdiv(nt, 1024 + 32));
  if (S > W) S = W;
  const int64_t fill = (int64_t)sm * 32 * 4 / 5;
  while (2 * S <= W && n * S * Sg < fill && cdiv(nt, 2 * S) >= 128) S *= 2;
  auto round_fill = [&](int s) {
    const int64_t RT = W / s, nr = cdiv(n, NCLS);
    int64_t C = (int64_t)sm * cps_warps / Sg;
    if (C > cdiv(nr, RT) * NCLS) C = cdiv(nr, RT) * NCLS;
    C = C / NCLS * NCLS;
    if (C < NCLS) C = NCLS;
    const int64_t Cq = C / NCLS;
    return ((double)nr / (double)Cq) / (double)(cdiv(cdiv(nr, Cq), RT) * RT);
  };
  while (2 * S <= W && cdiv(nt, 2 * S) >= 128 && round_fill(S) < 0.75 && round_fill(2 * S) > round_fill(S)) S *= 2;
  return S;
}

// Rows split over several warps with 8 loads per lane: two rows per warp
// with twice the split instead (same rows per tile, same bytes in flight,
// half as many shared-memory reads of a per byte of B; slices still of 128
// blocks or more).  Measured on GB300 as gemv() launches them, two
// repeats: faster on all 11 sweep shapes where it applies (7168 x 16384
// 34.06 -> 33.27 us, 4096 x 14336 19.49 -> 18.69, 4099 x 16384 21.85 ->
// 20.67, 256 x 262144 24.61 -> 23.38, 65536 x 16384 294.9 -> 294.0).
// Returns true (and updates S, R, U) when it applies.
bool two_rows_per_warp(int64_t nt, int W, int &S, int &R, int &U) {
  if (S < 2 || U != 8 || 2 * S > W || cdiv(nt, 2 * S) < 128) return false;
  S *= 2;
  R = 2;
  U = 4;
  return true;
}

// Planner of the tiles and bulk variants (pure host arithmetic).
//  * k-segments: as few as the shared-memory budget allows, more when the
//    rows alone cannot give every SM work (split-K).
//  * S (warps per row): tiles_split() for the tiles kernel; slices of about
//    512 blocks for the bulk kernel.  Tiles kernel: R = 2 rows per warp
//    side by side where every resident warp has two rows anyway.
//  * C (CTAs per segment): every SM busy at 32 resident warps (fewer when
//    shared memory limits the CTAs per SM), a multiple of 8 (one row class
//    per CTA) unless the rows are 16-byte aligned.
int plan_tiles(int64_t n, int64_t k, bool aligned, int sm, const gemv_config *f, gemv_config *out,
               bool bulk = false) {
  const int NCLS = aligned ? 1 : 8;
  const int W_list[3] = {16, 8, 4};
  // The tiles kernel runs 16-warp CTAs unless forced (measured best or
  // within 3 % on every workload shape); the bulk kernel, whose shared
  // memory limits it to one CTA per SM, tries smaller CTAs for small shapes.
  const int nW = (bulk && !f->warps_per_cta) ? 3 : 1;
  gemv_config best{};
  bool have = false;
  for (int wi = 0; wi < nW; ++wi) {
    const int W = f->warps_per_cta ? f->warps_per_cta : W_list[wi];
    if (!valid_W(W)) return GEMV_ERR_CONFIG;
    const int cps_warps = 32 / W;
    // k-segments
    int64_t Sg = f->grid_split ? f->grid_split : cdiv(k, kMaxSegment);
    if (Sg < 1 || Sg > kMaxSegments) return GEMV_ERR_CONFIG;
    int64_t kseg = (Sg == 1) ? k : round_up(cdiv(k, Sg), 8);
    Sg = cdiv(k, kseg);
    if (kseg > kMaxSegment) return GEMV_ERR_CONFIG;
    const int64_t nt_est = cdiv(kseg, 8) + (aligned ? 0 : 1);
    // slices and per-lane depth
    int S;
    if (f->warp_split) {
      S = f->warp_split;
      if (S < 1 || S > W || W % S != 0) return GEMV_ERR_CONFIG;
    } else if (!bulk) {
      S = tiles_split(n, nt_est, W, sm, Sg, NCLS, cps_warps);
    } else {
      // Bulk kernel: slices of about 512 blocks (two 4 KB ring chunks), so
      // that each warp's ring streams several chunks per row (a whole row
      // per warp measured up to 8 % slower at k = 7168).
      const int64_t q = (nt_est + 256) / 512;  // nt_est / 512, rounded
      S = (int)pow2_floor(q < 1 ? 1 : q);
      if (2 * S <= W && nt_est > 3 * S * 512 / 2) S *= 2;  // round up past 1.5x
      if (S > W) S = W;
      // Too few row tiles to occupy every CTA: split rows further while a
      // slice keeps at least 4 loads per lane.
      const int64_t resident_est = (int64_t)sm * cps_warps;
      while (S < W && nt_est / (2 * S) >= 128 &&
             cdiv(cdiv(n, NCLS), (int64_t)(W / S)) * NCLS < resident_est) {
        S *= 2;
      }
    }
    int R, U;
    if (bulk) {
      // One row per warp; a ring buffer is 32 * U blocks.
      if (f->rows_per_warp > 1) return GEMV_ERR_CONFIG;
      R = 1;
      U = f->unroll ? f->unroll : (cdiv(nt_est, S) <= 128 ? 4 : 8);
      if (U != 4 && U != 8) return GEMV_ERR_CONFIG;
    } else if (f->rows_per_warp || f->unroll) {
      R = f->rows_per_warp ? f->rows_per_warp : 1;
      U = f->unroll ? f->unroll : (R == 1 ? 8 : (R == 2 ? 4 : 2));
      if (!valid_tiles_RU(R, U)) return GEMV_ERR_CONFIG;
    } else {
      R = 1;
      U = cdiv(nt_est, S) <= 128 ? 4 : 8;
      // Two rows per warp (four loads each, so a staged vector of a serves
      // both) where every resident warp has two rows or more anyway and the
      // last round of row tiles wastes no more warp slots than with one:
      // 18432 x 7168 40.5 -> 38.6 us, 65536 x 4096 77.2 -> 76.4 us.
      if (S == 1 && n >= 2LL * sm * 32) {
        const int64_t nr = cdiv(n, NCLS);
        auto round_fill = [&](int64_t RT) {
          int64_t C = (int64_t)sm * cps_warps / Sg;
          if (C > cdiv(nr, RT) * NCLS) C = cdiv(nr, RT) * NCLS;
          C = C / NCLS * NCLS;
          if (C < NCLS) C = NCLS;
          const int64_t Cq = C / NCLS;
          const int64_t rounds = cdiv(cdiv(nr, Cq), RT);
          return ((double)nr / (double)Cq) / (double)(rounds * RT);
        };
        if (round_fill(2LL * W) >= 0.99 * round_fill(W)) {
          R = 2;
          U = 4;
          // Rows of 1024 blocks or more (k >= 8192; S = 1 allows up to
          // 1056): two warps per pair of rows, slices of whole 128-block
          // steps (28672 x 8192 bf16 65.05 -> 63.85 us as gemv() launches
          // it; at 896 blocks the halves are 3.5 steps and it was slower:
          // 18432 x 7168 36.6 -> 36.9 us).
          if (!f->warp_split && nt_est >= 1024 && 2 <= W) S = 2;
        }
      } else if (!f->warp_split) {
        two_rows_per_warp(nt_est, W, S, R, U);
      }
    }
    // row tiles and grid
    int64_t RT = (int64_t)(W / S) * R;
    const int64_t rows_per_class = cdiv(n, NCLS);
    int64_t groups = cdiv(rows_per_class, RT);  // tiles per class per segment
    const int64_t as_elems = round_up(kseg + 24, 8);
    int NS = 0;  // bulk: ring buffers per warp
    if (bulk) {
      if (f->stages) {
        NS = f->stages;
        if (NS < 2 || NS > 8) return GEMV_ERR_CONFIG;
      } else {
        // Two buffers per warp: 16 warps x 2 x 4 KiB in flight per SM, as
        // many bytes as the register kernel keeps in flight.  Deeper rings
        // measured slower on GB300 (7168 x 16384: 36.3 us with 2, 36.7 with
        // 3; 28672 x 8192: 66.6 vs 70.1 us).
        NS = kBulkDefaultStages;
      }
    } else if (f->stages) {
      return GEMV_ERR_CONFIG;
    }
    const int64_t smem = bulk ? bulk_smem_bytes(as_elems, W, U, NS) : as_elems * 2 + 2LL * W * R * 4;
    if (smem > kMaxSmemPerCta) return GEMV_ERR_CONFIG;
    int cps = cps_warps;
    const int64_t cps_smem = kSmemPerSm / (smem + kSmemReservedPerCta);
    if (cps_smem < cps) cps = (int)cps_smem;
    if (cps < 1) return GEMV_ERR_CONFIG;
    const int64_t resident = (int64_t)sm * cps;
    // Few rows and long rows: split k across CTAs so that every SM works.
    if (!f->grid_split && groups * NCLS * Sg < resident / 2) {
      const int64_t more = resident / (groups * NCLS);
      const int64_t max_by_k = cdiv(k, 256 * 8) > 1 ? cdiv(k, 256 * 8) : 1;
      int64_t Sg2 = more < max_by_k ? more : max_by_k;
      if (Sg2 > kMaxGridSplit) Sg2 = kMaxGridSplit;
      if (Sg2 > Sg) {
        Sg = Sg2;
        kseg = round_up(cdiv(k, Sg), 8);
        Sg = cdiv(k, kseg);
        // The segments are shorter now: choose the tiles kernel's split for
        // their length (few rows: R = 1 in any case).
        if (!bulk && !f->warp_split && !f->rows_per_warp && !f->unroll) {
          const int64_t nt2 = cdiv(kseg, 8) + (aligned ? 0 : 1);
          S = tiles_split(n, nt2, W, sm, Sg, NCLS, cps_warps);
          R = 1;
          U = cdiv(nt2, S) <= 128 ? 4 : 8;
          two_rows_per_warp(nt2, W, S, R, U);
          RT = (int64_t)(W / S) * R;
          groups = cdiv(rows_per_class, RT);
        }
      }
    }
    int64_t C;
    if (f->ctas) {
      C = (f->ctas / Sg) / NCLS * NCLS;
    } else {
      C = resident / Sg;
      const int64_t need = groups * NCLS;  // CTAs that would have work in whole tiles
      // Rows are dealt to a class's CTAs one at a time, so a grid of every
      // resident slot still gives each CTA rows, in one part-filled tile
      // instead of fewer CTAs with full ones.  Kept for the tiles kernel
      // when each CTA gets at least half a tile and rows are long: measured
      // on GB300 as gemv() launches it, 1024 x 16384 f16 7.96 -> 7.74 us,
      // 4099 x 7169 bf16 11.50 -> 11.32, 4099 x 4096 f16 7.25 -> 7.15,
      // 4096 x 4096 bf16 7.16 -> 7.10, others within 0.5 %; at k = 1000 it
      // was slower (4099 x 1000 3.38 -> 3.43, 1024 x 1000 2.81 -> 3.21).
      const bool spread = !bulk && Sg == 1 && k >= 4096 && C / NCLS >= 1 &&
                          rows_per_class * 2 >= RT * (C / NCLS);
      if (C > need && !spread) C = need;
      C = C / NCLS * NCLS;
    }
    if (C < NCLS) C = NCLS;
    if (C * Sg > INT32_MAX) return GEMV_ERR_CONFIG;

    gemv_config c{};
    c.variant = bulk ? GEMV_VARIANT_BULK : GEMV_VARIANT_TILES;
    c.rows_per_warp = R;
    c.unroll = U;
    c.warps_per_cta = W;
    c.warp_split = S;
    c.grid_split = (int32_t)Sg;
    c.row_blocks = (int32_t)C;
    c.ctas = (int32_t)(C * Sg);
    c.smem_bytes = (int32_t)(bulk ? bulk_smem_bytes(round_up(kseg + 24, 8), W, U, NS)
                                  : round_up(kseg + 24, 8) * 2 + 2LL * W * R * 4);
    c.stages = NS;
    c.launches = Sg > 1 ? 2 : 1;
    c.k_segment = kseg;
    if (f->l2_prefetch) {
      if (f->l2_prefetch < -1 || f->l2_prefetch > 3 || (bulk && f->l2_prefetch > 0)) return GEMV_ERR_CONFIG;
      c.l2_prefetch = f->l2_prefetch < 0 ? 0 : f->l2_prefetch;
    } else {
      c.l2_prefetch = kDefaultL2Prefetch;
    }
    best = c;
    have = true;
    if (f->warps_per_cta || c.ctas >= sm) break;
  }
  if (!have) return GEMV_ERR_CONFIG;
  *out = best;
  return GEMV_OK;
}

bool is_unforced(const gemv_config &f) {
  return !(f.variant || f.rows_per_warp || f.warps_per_cta || f.warp_split || f.grid_split || f.ctas ||
           f.unroll || f.l2_prefetch || f.stages);
}

// The planner.  Pure host arithmetic: no CUDA call.
int plan_impl(int64_t n, int64_t k, int dtype, bool aligned, int sm, const gemv_config *f,
              gemv_config *out) {
  if (dtype < 0 || dtype > 3) return GEMV_ERR_DTYPE;
  if (n < 1 || k < 1 || k > INT32_MAX || sm < 1) return GEMV_ERR_ARG;
  gemv_config fz{};
  if (f == nullptr || is_unforced(*f)) f = &fz;

  const int auto_variant = (kAutoVariant == GEMV_VARIANT_ROWS && !aligned) ? GEMV_VARIANT_ROWS_GENERAL
                                                                            : kAutoVariant;
  const int variant = f->variant ? f->variant : auto_variant;
  if (variant == GEMV_VARIANT_TILES && f == &fz) {
    // Nothing forced: the tiles plan, or the bulk variant where it measured
    // at least as fast on GB300: B of 768 MiB or more whose tiles plan
    // streams each row with one warp, with rows of 6144 to 8191 elements.
    // There (57344 x 7168, 65536 x 7169) the two are equal back to back as
    // gemv() launches them, and the bulk kernel is 1-2 % faster as plain
    // and as isolated launches (65536 x 7169 under ncu: 85.1 % of the DRAM
    // peak against 80.8 %).  With shorter rows the tiles kernel, which
    // stages a ahead of its first loads, is 2-4 % faster back to back
    // (131072 x 4096 151.6 -> 145.5 us, 262144 x 2048 150.2 -> 145.1), and
    // at k = 8192 on three of four shapes (57344 x 8192 130.2 -> 127.1).
    int st = plan_tiles(n, k, aligned, sm, f, out);
    const int64_t b_bytes = n * k * 2;
    if (st == GEMV_OK && out->warp_split <= out->rows_per_warp && b_bytes >= kBulkAutoBytes &&
        k >= kBulkAutoMinK && k < kBulkAutoEndK) {
      gemv_config b{};
      if (plan_tiles(n, k, aligned, sm, f, &b, true) == GEMV_OK) *out = b;
    }
    return st;
  }
  if (variant == GEMV_VARIANT_TILES) return plan_tiles(n, k, aligned, sm, f, out);
  if (variant == GEMV_VARIANT_BULK) return plan_tiles(n, k, aligned, sm, f, out, true);
  if (f->stages) return GEMV_ERR_CONFIG;
  if (variant != GEMV_VARIANT_ROWS && variant != GEMV_VARIANT_ROWS_GENERAL) return GEMV_ERR_CONFIG;
  if (variant == GEMV_VARIANT_ROWS && !aligned) return GEMV_ERR_CONFIG;

  const int64_t nt = cdiv(k, 8);  // 16-byte vectors per row
  const int64_t warp_slots = (int64_t)sm * 32;  // 32 resident warps per SM
  int R;
  if (f->rows_per_warp) {
    R = f->rows_per_warp;
    if (!valid_R(R)) return GEMV_ERR_CONFIG;
  } else if (variant == GEMV_VARIANT_ROWS_GENERAL) {
    R = 1;
  } else if (n >= warp_slots * 4 && k * 2 <= 2048) {
    R = 4;
  } else if (n >= warp_slots * 2 && k * 2 <= 8192) {
    R = 2;
  } else {
    R = 1;
  }
  if (variant == GEMV_VARIANT_ROWS_GENERAL && R != 1) return GEMV_ERR_CONFIG;

  const int64_t row_groups = cdiv(n, R);
  // Splits of a row needed so that every warp slot of the GPU has work, and
  // the most that still leave every lane at least two 16-byte loads.
  const int64_t want = row_groups >= warp_slots ? 1 : cdiv(warp_slots, row_groups);
  const int64_t max_split = nt / 64 > 1 ? nt / 64 : 1;
  const int64_t split = want < max_split ? want : max_split;

  gemv_config best{};
  bool have = false;
  const int W_list[3] = {16, 8, 4};
  for (int wi = 0; wi < 3; ++wi) {
    const int W = f->warps_per_cta ? f->warps_per_cta : W_list[wi];
    if (!valid_W(W)) return GEMV_ERR_CONFIG;
    int Sw;
    if (f->warp_split) {
      Sw = f->warp_split;
      if (Sw < 1 || Sw > W || W % Sw != 0) return GEMV_ERR_CONFIG;
    } else {
      Sw = (int)(pow2_floor(split) < W ? pow2_floor(split) : W);
    }
    int64_t Sg;
    if (f->grid_split) {
      Sg = f->grid_split;
      if (Sg < 1 || Sg > kMaxSegments) return GEMV_ERR_CONFIG;
    } else {
      Sg = cdiv(k, kMaxSegment);
      const int64_t need = split > Sw ? cdiv(split, Sw) : 1;
      if (need > Sg) Sg = need > kMaxGridSplit ? (Sg > kMaxGridSplit ? Sg : kMaxGridSplit) : need;
      // a forced CTA count caps the split (but not below what k requires)
      if (f->ctas && Sg > f->ctas) Sg = f->ctas > cdiv(k, kMaxSegment) ? f->ctas : cdiv(k, kMaxSegment);
    }
    int64_t kseg = (Sg == 1) ? k : round_up(cdiv(k, Sg), 8);
    Sg = cdiv(k, kseg);  // every segment non-empty
    if (kseg > kMaxSegment) return GEMV_ERR_CONFIG;

    // CTAs resident per SM: 32 warps by the kernel's register bound (at most
    // 64 registers a thread), fewer if shared memory runs out first.
    int cps = 32 / W;
    const int64_t as_elems = round_up(kseg + 24, 8);
    const int64_t smem = as_elems * 2 + (int64_t)W * R * 4;
    if (smem > kMaxSmemPerCta) return GEMV_ERR_CONFIG;
    const int64_t cps_smem = kSmemPerSm / (smem + kSmemReservedPerCta);
    if (cps_smem < cps) cps = (int)cps_smem;
    const int64_t slots = W / Sw;
    const int64_t max_rb = ((int64_t)sm * cps) / Sg > 0 ? ((int64_t)sm * cps) / Sg : 1;
    int64_t nrb;
    if (f->ctas) {
      if (f->ctas < Sg) return GEMV_ERR_CONFIG;
      nrb = f->ctas / Sg;
    } else {
      nrb = cdiv(n, slots * R);
      if (nrb > max_rb) nrb = max_rb;
    }
    if (nrb * Sg > INT32_MAX) return GEMV_ERR_CONFIG;

    gemv_config c{};
    c.variant = variant;
    c.rows_per_warp = R;
    c.warps_per_cta = W;
    c.warp_split = Sw;
    c.grid_split = (int32_t)Sg;
    c.row_blocks = (int32_t)nrb;
    c.ctas = (int32_t)(nrb * Sg);
    c.smem_bytes = (int32_t)smem;
    c.launches = Sg > 1 ? 2 : 1;
    c.k_segment = kseg;
    c.unroll = unroll_for_rows(R);
    best = c;
    have = true;
    // Prefer big CTAs unless that leaves SMs idle; a forced W ends the search.
    if (f->warps_per_cta || c.ctas >= sm) break;
  }
  if (!have) return GEMV_ERR_CONFIG;
  *out = best;
  return GEMV_OK;
}

MainKernel lookup_main(int dtype, const gemv_config &c, bool aligned, bool epi = false) {
  const int of = dtype >= 2 ? 1 : 0;
  if (c.variant == GEMV_VARIANT_TILES) {
    return (dtype & 1) ? tiles_kernel_bf16(of, aligned ? 1 : 0, c.rows_per_warp, c.unroll, epi ? 1 : 0)
                       : tiles_kernel_f16(of, aligned ? 1 : 0, c.rows_per_warp, c.unroll, epi ? 1 : 0);
  }
  if (c.variant == GEMV_VARIANT_BULK) {
    return (dtype & 1) ? bulk_kernel_bf16(of, aligned ? 1 : 0, c.unroll, epi ? 1 : 0)
                       : bulk_kernel_f16(of, aligned ? 1 : 0, c.unroll, epi ? 1 : 0);
  }
  return (dtype & 1) ? main_kernel_bf16(of, c.variant, c.rows_per_warp)
                     : main_kernel_f16(of, c.variant, c.rows_per_warp);
}

ReduceKernel lookup_reduce(int dtype) {
  const int of = dtype >= 2 ? 1 : 0;
  return (dtype & 1) ? reduce_kernel_bf16(of) : reduce_kernel_f16(of);
}

// Opt a kernel into more than 48 KiB of dynamic shared memory on this
// device, once (caller holds g_mu).
cudaError_t ensure_smem_attr_locked(const void *fn, int dev, int smem) {
  if (smem <= 48 * 1024) return cudaSuccess;
  auto key = std::make_pair(fn, dev);
  if (g_func_attr_set.count(key)) return cudaSuccess;
  cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, kMaxSmemPerCta);
  if (e == cudaSuccess) g_func_attr_set.insert(key);
  return e;
}

// Workspace of at least `bytes` for (dev, stream) (caller holds g_mu).
int workspace_locked(int dev, cudaStream_t stream, size_t bytes, float **out) {
  Workspace &w = g_ws[std::make_pair(dev, stream)];
  if (w.bytes < bytes) {
    if (w.ptr) {
      // The previous buffer may still be in use by work queued on `stream`.
      cudaError_t e = cudaStreamSynchronize(stream);
      if (e != cudaSuccess) return cuda_fail(e);
      cudaFree(w.ptr);
      w.ptr = nullptr;
      w.bytes = 0;
    }
    void *p = nullptr;
    if (cudaMalloc(&p, bytes) != cudaSuccess) {
      cudaGetLastError();
      return GEMV_ERR_NOMEM;
    }
    w.ptr = static_cast<float *>(p);
    w.bytes = bytes;
  }
  *out = w.ptr;
  return GEMV_OK;
}

bool overlaps(const void *p, int64_t pbytes, const void *q, int64_t qbytes) {
  const uintptr_t a0 = (uintptr_t)p, a1 = a0 + (uintptr_t)pbytes;
  const uintptr_t b0 = (uintptr_t)q, b1 = b0 + (uintptr_t)qbytes;
  return a0 < b1 && b0 < a1;
}

// Checks that need no CUDA call (row stride ldb >= k).  Returns GEMV_OK or
// an error; n == 0 passes (nothing will be launched).
int validate_ld(const void *B, int64_t ldb, const void *a, const void *c, int64_t n, int64_t k, int dtype) {
  if (dtype < 0 || dtype > 3) return GEMV_ERR_DTYPE;
  if (n < 0 || k < 0 || k > INT32_MAX) return GEMV_ERR_ARG;
  if (ldb < k || ldb > INT32_MAX) return GEMV_ERR_ARG;
  if (n == 0) return GEMV_OK;
  if (c == nullptr) return GEMV_ERR_ARG;
  if (k > 0 && (B == nullptr || a == nullptr)) return GEMV_ERR_ARG;
  const int oe = out_elem_bytes(dtype);
  if (((uintptr_t)c % (uintptr_t)oe) != 0) return GEMV_ERR_ALIGN;
  if (k > 0 && (((uintptr_t)B & 1u) || ((uintptr_t)a & 1u))) return GEMV_ERR_ALIGN;
  if (n > INT64_MAX / (ldb > 0 ? ldb : 1) / 2) return GEMV_ERR_ARG;
  if (k > 0) {
    const int64_t cb = n * oe;
    const int64_t bb = ((n - 1) * ldb + k) * 2;
    if (overlaps(c, cb, B, bb) || overlaps(c, cb, a, k * 2)) return GEMV_ERR_ALIAS;
  }
  return GEMV_OK;
}

int validate(const void *B, const void *a, const void *c, int64_t n, int64_t k, int dtype) {
  return validate_ld(B, k, a, c, n, k, dtype);
}

Epilogue identity_epilogue() {
  Epilogue ep;
  ep.alpha = 1.f;
  ep.beta = 0.f;
  ep.bias = nullptr;
  ep.bias_f32 = 0;
  ep.act = GEMV_ACT_NONE;
  return ep;
}

bool is_identity(const Epilogue &ep) {
  return ep.alpha == 1.f && ep.bias == nullptr && ep.act == GEMV_ACT_NONE;
}

// Device address of the timeout counter on `dev` (the current device),
// looked up once per device.
int timeout_counter(int dev, uint32_t **out) {
  std::lock_guard<std::mutex> lk(g_mu);
  if (g_timeouts_ptr[dev] == nullptr) {
    void *p = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&p, g_gemv_wait_timeouts);
    if (e != cudaSuccess || p == nullptr) {
      cudaGetLastError();
      return cuda_fail(e != cudaSuccess ? e : cudaErrorInvalidSymbol);
    }
    g_timeouts_ptr[dev] = static_cast<uint32_t *>(p);
  }
  *out = g_timeouts_ptr[dev];
  return GEMV_OK;
}

int run_ld(const void *B, int64_t ldb, const void *a, void *c, int64_t n, int64_t k, int dtype,
           const gemv_config *forced, const Epilogue &ep, cudaStream_t stream) {
  int inj = g_inject.exchange(0);
  if (inj != 0) return inj;
  int st = validate_ld(B, ldb, a, c, n, k, dtype);
  if (st != GEMV_OK) return st;
  if (n == 0) return GEMV_OK;

  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    cudaGetLastError();
    return GEMV_ERR_DEVICE;
  }
  if (!on_device(dev, {k > 0 ? B : nullptr, k > 0 ? a : nullptr, c, ep.bias})) return GEMV_ERR_DEVICE;
  if (k == 0) {
    // The empty sum: +0 in every output format is all-zero bits; with an
    // epilogue, its value on 0 (the second-pass kernel over no partials).
    if (is_identity(ep)) {
      e = cudaMemsetAsync(c, 0, (size_t)n * out_elem_bytes(dtype), stream);
    } else {
      ReduceKernel rk = lookup_reduce(dtype);
      rk<<<reduce_blocks(n, 0), kReduceThreads, 0, stream>>>(nullptr, c, n, 0, ep);
      e = cudaGetLastError();
    }
    if (e != cudaSuccess) return cuda_fail(e);
    gemv_config z{};
    t_last = z;
    t_has_last = true;
    return GEMV_OK;
  }
  const bool aligned = (((uintptr_t)B & 15u) == 0) && (k % 8 == 0) && (ldb % 8 == 0);
  // Without a configuration the launch is a programmatic dependent launch
  // that touches no memory before the predecessor has completed
  // (GEMV_OVERLAP_PDL): always safe, and 1.5-2.3 us per call faster back to
  // back on GB300 than a plain launch.
  const int overlap = forced ? forced->overlap : GEMV_OVERLAP_PDL;
  if (overlap < GEMV_OVERLAP_NONE || overlap > GEMV_OVERLAP_PDL_PREFETCH_BA) return GEMV_ERR_CONFIG;

  gemv_config cfg{};
  float *ws = nullptr;
  MainKernel mk = nullptr;
  bool defer = false;        // keep row results in shared memory, store after one wait
  int64_t launch_smem = 0;   // dynamic shared memory of the launch
  {
    std::lock_guard<std::mutex> lk(g_mu);
    const DeviceInfo &di = device_info_locked(dev);
    if (!di.ok) return GEMV_ERR_DEVICE;
    const bool is_forced = forced != nullptr && (forced->variant || forced->rows_per_warp ||
                                                 forced->warps_per_cta || forced->warp_split ||
                                                 forced->grid_split || forced->ctas || forced->unroll ||
                                                 forced->l2_prefetch || forced->stages);
    if (is_forced) {
      st = plan_impl(n, k, dtype, aligned, di.sm_count, forced, &cfg);
      if (st != GEMV_OK) return st;
    } else {
      Key key{dev, dtype, aligned ? 1 : 0, n, k};
      auto it = g_cache.find(key);
      if (it != g_cache.end()) {
        cfg = it->second;
      } else {
        st = plan_impl(n, k, dtype, aligned, di.sm_count, nullptr, &cfg);
        if (st != GEMV_OK) return st;
        g_cache.emplace(key, cfg);
        log_config("new config", dev, n, k, dtype, aligned, cfg);
      }
    }
    launch_smem = cfg.smem_bytes;
    if (cfg.smem_bytes > di.max_smem_optin) return GEMV_ERR_CONFIG;
    // Shared input vector promised (B and a unwritten by the work in
    // flight): the tiles kernel keeps its row results (at most
    // kDeferMaxRows per CTA) and writes them after one wait at the end, so
    // it streams all of B while the preceding kernel drains.
    if (overlap == GEMV_OVERLAP_PDL_PREFETCH_BA && cfg.variant == GEMV_VARIANT_TILES) {
      const int NCLS = aligned ? 1 : 8;
      const int64_t nloc_max = cdiv(cdiv(n, NCLS), (int64_t)cfg.row_blocks / NCLS);
      const int64_t extra = round_up(nloc_max * 4, 16);
      if (nloc_max <= kDeferMaxRows && cfg.smem_bytes + extra <= di.max_smem_optin) {
        defer = true;
        launch_smem = cfg.smem_bytes + extra;
      }
    }
    mk = lookup_main(dtype, cfg, aligned, !is_identity(ep));
    if (mk == nullptr) return GEMV_ERR_CONFIG;
    e = ensure_smem_attr_locked((const void *)mk, dev, (int)launch_smem);
    if (e != cudaSuccess) return cuda_fail(e);
    if (cfg.grid_split > 1) {
      st = workspace_locked(dev, stream, (size_t)cfg.grid_split * (size_t)n * sizeof(float), &ws);
      if (st != GEMV_OK) return st;
    }
  }

  Params p;
  p.B = static_cast<const uint16_t *>(B);
  p.a = static_cast<const uint16_t *>(a);
  p.c = c;
  p.ws = ws;
  p.n = n;
  p.k = k;
  p.ldb = ldb;
  p.kseg = cfg.k_segment;
  p.base_off = (int32_t)(((uintptr_t)B >> 1) & 7u);
  p.sg = cfg.grid_split;
  p.sw = cfg.warp_split;
  p.nrb = cfg.row_blocks;
  p.as_elems = (int32_t)round_up(cfg.k_segment + 24, 8);
  p.ep = ep;
  p.stages = cfg.stages;
  p.wait_polls = kWaitPolls;
  p.timeouts = nullptr;
  if (cfg.variant == GEMV_VARIANT_BULK) {
    st = timeout_counter(dev, &p.timeouts);
    if (st != GEMV_OK) return st;
    const int budget = g_wait_budget.exchange(-1);
    if (budget >= 0) p.wait_polls = budget;
  }
  p.flags = ((overlap >= GEMV_OVERLAP_PDL_PREFETCH_B) ? kFlagPrefetchB : 0) |
            ((overlap == GEMV_OVERLAP_PDL_PREFETCH_BA) ? kFlagPrefetchA : 0) |
            (is_identity(ep) ? 0 : kFlagEpilogue) | (defer ? kFlagDeferStores : 0) |
            ((overlap == GEMV_OVERLAP_PDL) ? kFlagL2First : 0) | (cfg.l2_prefetch << kFlagL2Shift);

  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t lc = {};
  lc.gridDim = dim3((unsigned)cfg.ctas);
  lc.blockDim = dim3((unsigned)(cfg.warps_per_cta * 32));
  lc.dynamicSmemBytes = (size_t)launch_smem;
  lc.stream = stream;
  lc.attrs = attr;
  lc.numAttrs = overlap != GEMV_OVERLAP_NONE ? 1 : 0;
  e = cudaLaunchKernelEx(&lc, mk, p);
  if (e != cudaSuccess) return cuda_fail(e);
  if (cfg.grid_split > 1) {
    ReduceKernel rk = lookup_reduce(dtype);
    lc.gridDim = dim3(reduce_blocks(n, cfg.grid_split));
    lc.blockDim = dim3(kReduceThreads);
    lc.dynamicSmemBytes = 0;
    const float *wsc = ws;
    e = cudaLaunchKernelEx(&lc, rk, wsc, c, n, (int32_t)cfg.grid_split, ep);
    if (e != cudaSuccess) return cuda_fail(e);
  }
  cfg.overlap = overlap;
  t_last = cfg;
  t_has_last = true;
  return GEMV_OK;
}

int run(const void *B, const void *a, void *c, int64_t n, int64_t k, int dtype, const gemv_config *forced,
        cudaStream_t stream) {
  return run_ld(B, k, a, c, n, k, dtype, forced, identity_epilogue(), stream);
}

}  // namespace
}  // namespace gemvk

using namespace gemvk;

extern "C" int gemv(const void *B, const void *a, void *c, int64_t n, int64_t k, int dtype,
                    cudaStream_t stream) {
  return run(B, a, c, n, k, dtype, nullptr, stream);
}

extern "C" int gemv_ex(const void *B, const void *a, void *c, int64_t n, int64_t k, int dtype,
                       const gemv_config *forced, cudaStream_t stream) {
  return run(B, a, c, n, k, dtype, forced, stream);
}

extern "C" int gemv_fused(const void *B, int64_t ldb, const void *a, void *c, int64_t n, int64_t k, int dtype,
                          const gemv_epilogue *epilogue, const gemv_config *config, cudaStream_t stream) {
  Epilogue ep = identity_epilogue();
  if (epilogue != nullptr) {
    if (epilogue->activation < GEMV_ACT_NONE || epilogue->activation > GEMV_ACT_SILU) return GEMV_ERR_ARG;
    if (epilogue->bias_dtype != GEMV_BIAS_INPUT_TYPE && epilogue->bias_dtype != GEMV_BIAS_F32) return GEMV_ERR_ARG;
    ep.alpha = epilogue->alpha;
    ep.beta = epilogue->beta;
    ep.bias = epilogue->bias;
    ep.bias_f32 = epilogue->bias_dtype == GEMV_BIAS_F32 ? 1 : 0;
    ep.act = epilogue->activation;
    if (ep.bias != nullptr && n > 0) {
      const int be = ep.bias_f32 ? 4 : 2;
      if ((uintptr_t)ep.bias % (uintptr_t)be != 0) return GEMV_ERR_ALIGN;
      if (c != nullptr && overlaps(c, n * out_elem_bytes(dtype), ep.bias, n * be)) return GEMV_ERR_ALIAS;
    }
  }
  return run_ld(B, ldb, a, c, n, k, dtype, config, ep, stream);
}

extern "C" int gemv_plan(int64_t n, int64_t k, int dtype, int b_aligned16, int sm_count,
                         const gemv_config *forced, gemv_config *out) {
  if (out == nullptr) return GEMV_ERR_ARG;
  const bool aligned = b_aligned16 != 0 && k % 8 == 0;
  const int st = plan_impl(n, k, dtype, aligned, sm_count, forced, out);
  if (st == GEMV_OK) log_config("plan", -1, n, k, dtype, aligned, *out);
  return st;
}

extern "C" int gemv_prepare(int64_t n, int64_t k, int dtype, int b_aligned16, cudaStream_t stream) {
  if (dtype < 0 || dtype > 3) return GEMV_ERR_DTYPE;
  if (n < 0 || k < 0 || k > INT32_MAX) return GEMV_ERR_ARG;
  if (n == 0 || k == 0) return GEMV_OK;
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    cudaGetLastError();
    return GEMV_ERR_DEVICE;
  }
  const bool aligned = b_aligned16 != 0 && k % 8 == 0;
  std::lock_guard<std::mutex> lk(g_mu);
  const DeviceInfo &di = device_info_locked(dev);
  if (!di.ok) return GEMV_ERR_DEVICE;
  Key key{dev, dtype, aligned ? 1 : 0, n, k};
  gemv_config cfg{};
  auto it = g_cache.find(key);
  if (it != g_cache.end()) {
    cfg = it->second;
  } else {
    int st = plan_impl(n, k, dtype, aligned, di.sm_count, nullptr, &cfg);
    if (st != GEMV_OK) return st;
    g_cache.emplace(key, cfg);
    log_config("new config", dev, n, k, dtype, aligned, cfg);
  }
  MainKernel mk = lookup_main(dtype, cfg, aligned);
  if (mk == nullptr) return GEMV_ERR_CONFIG;
  cudaError_t e = ensure_smem_attr_locked((const void *)mk, dev, cfg.smem_bytes);
  if (e != cudaSuccess) return cuda_fail(e);
  if (cfg.grid_split > 1) {
    float *ws = nullptr;
    return workspace_locked(dev, stream, (size_t)cfg.grid_split * (size_t)n * sizeof(float), &ws);
  }
  return GEMV_OK;
}

extern "C" int gemv_last_config(gemv_config *out) {
  if (out == nullptr) return GEMV_ERR_ARG;
  if (!t_has_last) return GEMV_ERR_ARG;
  *out = t_last;
  return GEMV_OK;
}

extern "C" const char *gemv_status_string(int status) {
  switch (status) {
    case GEMV_OK: return "ok";
    case GEMV_ERR_ARG: return "invalid argument (null pointer, negative or oversized n/k)";
    case GEMV_ERR_DTYPE: return "unknown dtype code";
    case GEMV_ERR_ALIAS: return "output c overlaps input B or a";
    case GEMV_ERR_DEVICE:
      return "no usable device (current device must be sm_103), or a buffer not in the current device's memory";
    case GEMV_ERR_CUDA: return "a CUDA call or kernel launch failed (see gemv_last_cuda_error)";
    case GEMV_ERR_CONFIG: return "configuration invalid for this shape";
    case GEMV_ERR_ALIGN: return "pointer not aligned to its element type";
    case GEMV_ERR_NOMEM: return "split-K workspace allocation failed";
    case GEMV_ERR_SCRATCH: return "split-K scratch needed (segments * n floats) exceeds the static scratch array";
    default: return "unknown status";
  }
}

extern "C" int gemv_last_cuda_error(void) { return t_cuda_err; }

extern "C" int gemv_debug_inject(int status) {
  g_inject.store(status);
  return GEMV_OK;
}

extern "C" int gemv_debug_wait_budget(int32_t polls) {
  if (polls < -1) return GEMV_ERR_ARG;
  g_wait_budget.store(polls);
  return GEMV_OK;
}

extern "C" int gemv_wait_timeouts(int reset, uint32_t *count) {
  if (count == nullptr) return GEMV_ERR_ARG;
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    cudaGetLastError();
    return GEMV_ERR_DEVICE;
  }
  uint32_t *ptr = nullptr;
  int st = timeout_counter(dev, &ptr);
  if (st != GEMV_OK) return st;
  e = cudaMemcpy(count, ptr, sizeof(uint32_t), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return cuda_fail(e);
  if (reset) {
    e = cudaMemset(ptr, 0, sizeof(uint32_t));
    if (e == cudaSuccess) e = cudaDeviceSynchronize();
    if (e != cudaSuccess) return cuda_fail(e);
  }
  return GEMV_OK;
}

extern "C" int gemv_release(void) {
  std::lock_guard<std::mutex> lk(g_mu);
  int cur = -1;
  cudaGetDevice(&cur);
  for (auto &kv : g_ws) {
    if (kv.second.ptr) {
      cudaSetDevice(kv.first.first);
      cudaFree(kv.second.ptr);
    }
  }
  if (cur >= 0) cudaSetDevice(cur);
  cudaGetLastError();
  g_ws.clear();
  g_cache.clear();
  return GEMV_OK;
}

extern "C" int gemv_host(const void *B_host, const void *a_host, void *c_host, void *B_dev, void *a_dev,
                         void *c_dev, int64_t n, int64_t k, int dtype, cudaStream_t stream) {
  int inj = g_inject.exchange(0);
  if (inj != 0) return inj;
  int st = validate(B_dev, a_dev, c_dev, n, k, dtype);
  if (st != GEMV_OK) return st;
  if (n == 0) return GEMV_OK;
  if (c_host == nullptr || (k > 0 && (B_host == nullptr || a_host == nullptr))) return GEMV_ERR_ARG;
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    cudaGetLastError();
    return GEMV_ERR_DEVICE;
  }
  if (!on_device(dev, {k > 0 ? B_dev : nullptr, k > 0 ? a_dev : nullptr, c_dev})) return GEMV_ERR_DEVICE;
  if (k > 0) {
    e = cudaMemcpyAsync(B_dev, B_host, (size_t)n * (size_t)k * 2, cudaMemcpyHostToDevice, stream);
    if (e != cudaSuccess) return cuda_fail(e);
    e = cudaMemcpyAsync(a_dev, a_host, (size_t)k * 2, cudaMemcpyHostToDevice, stream);
    if (e != cudaSuccess) return cuda_fail(e);
  }
  st = run(B_dev, a_dev, c_dev, n, k, dtype, nullptr, stream);
  if (st != GEMV_OK) return st;
  e = cudaMemcpyAsync(c_host, c_dev, (size_t)n * out_elem_bytes(dtype), cudaMemcpyDeviceToHost, stream);
  if (e != cudaSuccess) return cuda_fail(e);
  return GEMV_OK;
}

// --------------------------------------------------------------------------
// Split-K without any allocation: the scratch lives in a fixed device array.
//
// Some callers must not allocate device memory while they run: an inference
// engine's per-layer plugin code that is forbidden to call cudaMalloc during
// execution, a serving loop where cudaMalloc would synchronize the device and
// stall the other streams, or a process whose device memory is handed out up
// front by its own allocator.  gemv_splitk_noalloc() serves them: the
// split-K partial sums go to g_gemv_static_scratch, a file-scope device array
// that exists on every GPU that loads this library, for the life of the
// process.  The caller still passes B, a and c.
static __device__ __align__(256) float g_gemv_static_scratch[GEMV_STATIC_SCRATCH_FLOATS];

namespace gemvk {
namespace {

std::mutex g_static_mu;
float *g_static_scratch_ptr[kMaxDevices] = {};

// Device address of the static scratch array on `dev`, which must be the
// current device.  In host code the array's name is only a host-side stand-in,
// so the address is looked up once per device with cudaGetSymbolAddress.
int static_scratch_for(int dev, float **out) {
  std::lock_guard<std::mutex> lk(g_static_mu);
  if (g_static_scratch_ptr[dev] == nullptr) {
    void *p = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&p, g_gemv_static_scratch);
    if (e != cudaSuccess || p == nullptr) {
      cudaGetLastError();
      return cuda_fail(e != cudaSuccess ? e : cudaErrorInvalidSymbol);
    }
    g_static_scratch_ptr[dev] = static_cast<float *>(p);
  }
  *out = g_static_scratch_ptr[dev];
  return GEMV_OK;
}

}  // namespace
}  // namespace gemvk

extern "C" int gemv_splitk_noalloc(const void *B, const void *a, void *c, int64_t n, int64_t k, int dtype,
                                   int grid_split, cudaStream_t stream) {
  int st = validate(B, a, c, n, k, dtype);
  if (st != GEMV_OK) return st;
  if (grid_split < 2 || grid_split > kMaxGridSplit) return GEMV_ERR_CONFIG;
  if (n == 0) return GEMV_OK;
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    cudaGetLastError();
    return GEMV_ERR_DEVICE;
  }
  if (!on_device(dev, {k > 0 ? B : nullptr, k > 0 ? a : nullptr, c})) return GEMV_ERR_DEVICE;
  if (k == 0) {
    e = cudaMemsetAsync(c, 0, (size_t)n * out_elem_bytes(dtype), stream);
    return e == cudaSuccess ? GEMV_OK : cuda_fail(e);
  }
  const bool aligned = (((uintptr_t)B & 15u) == 0) && (k % 8 == 0);
  gemv_config cfg{};
  MainKernel mk = nullptr;
  {
    std::lock_guard<std::mutex> lk(g_mu);
    const DeviceInfo &di = device_info_locked(dev);
    if (!di.ok) return GEMV_ERR_DEVICE;
    gemv_config forced{};
    forced.variant = GEMV_VARIANT_TILES;
    // A segment stages at most kMaxSegment columns of a: longer rows take
    // as many segments as that needs, even beyond the requested split.
    const int64_t need = cdiv(k, kMaxSegment);
    forced.grid_split = (int32_t)(need > grid_split ? need : grid_split);
    st = plan_impl(n, k, dtype, aligned, di.sm_count, &forced, &cfg);
    if (st != GEMV_OK) return st;
    if (cfg.smem_bytes > di.max_smem_optin) return GEMV_ERR_CONFIG;
    mk = lookup_main(dtype, cfg, aligned);
    if (mk == nullptr) return GEMV_ERR_CONFIG;
    e = ensure_smem_attr_locked((const void *)mk, dev, cfg.smem_bytes);
    if (e != cudaSuccess) return cuda_fail(e);
  }
  // Only a plan of two or more segments keeps partials in the scratch; a
  // short k can leave a single segment, which writes c directly and needs
  // no scratch whatever n is.
  if (cfg.grid_split > 1 && (int64_t)cfg.grid_split * n > (int64_t)GEMV_STATIC_SCRATCH_FLOATS)
    return GEMV_ERR_SCRATCH;
  float *ws = nullptr;
  if (cfg.grid_split > 1) {
    st = static_scratch_for(dev, &ws);
    if (st != GEMV_OK) return st;
  }
  Params p;
  p.B = static_cast<const uint16_t *>(B);
  p.a = static_cast<const uint16_t *>(a);
  p.c = c;
  p.ws = ws;
  p.n = n;
  p.k = k;
  p.ldb = k;
  p.kseg = cfg.k_segment;
  p.base_off = (int32_t)(((uintptr_t)B >> 1) & 7u);
  p.sg = cfg.grid_split;
  p.sw = cfg.warp_split;
  p.nrb = cfg.row_blocks;
  p.as_elems = (int32_t)round_up(cfg.k_segment + 24, 8);
  p.flags = 0;
  p.ep = identity_epilogue();
  p.stages = 0;
  p.wait_polls = kWaitPolls;
  p.timeouts = nullptr;
  // Every (segment, row) partial is written by the first kernel before the
  // second reads it, so the scratch needs no clearing between calls.
  mk<<<cfg.ctas, cfg.warps_per_cta * 32, cfg.smem_bytes, stream>>>(p);
  e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e);
  if (cfg.grid_split > 1) {
    ReduceKernel rk = lookup_reduce(dtype);
    rk<<<reduce_blocks(n, cfg.grid_split), kReduceThreads, 0, stream>>>(ws, c, n, cfg.grid_split,
                                                                           identity_epilogue());
    e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(e);
  }
  t_last = cfg;
  t_has_last = true;
  return GEMV_OK;
}
