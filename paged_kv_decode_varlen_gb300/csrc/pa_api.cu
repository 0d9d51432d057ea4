// C ABI of libpa: host-side validation, launch planning and diagnostics.
// The arithmetic is in the kernel files; this file only checks arguments,
// decides the launch plan from the host copies of the batch metadata and
// enqueues the kernels on the caller's stream.
#include <math.h>
#include <stdarg.h>
#include <stdio.h>
#include <string.h>

#include <algorithm>
#include <cmath>
#include <atomic>
#include <mutex>
#include <memory>
#include <vector>

#include <cudaTypedefs.h>  // PFN_cuTensorMapEncodeTiled

#include "common.cuh"
#include "internal.h"
#include "pa.h"

namespace {

thread_local char g_msg[512] = "";
std::atomic<int64_t> g_launches{0};
std::atomic<int32_t> g_forced_ctas{0};
std::atomic<int32_t> g_prefill_ctas{0};  // pa_set_prefill_ctas: > 0 forced, -1 never, 0 automatic
std::atomic<int32_t> g_decode_fault{0};  // pa_set_decode_fault_injection

pa_status fail(pa_status s, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_msg, sizeof g_msg, fmt, ap);
  va_end(ap);
  return s;
}

pa_status ok() {
  g_msg[0] = '\0';
  return PA_OK;
}

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// ------------------------------------------------------------------ trace
constexpr int kTraceCap = 16384;
struct TraceRec {
  int32_t kind;
  cudaEvent_t begin, end;
};
std::mutex g_trace_mu;
bool g_trace_on = false;
std::vector<TraceRec> g_trace;       // recorded, not yet read
std::vector<cudaEvent_t> g_evpool;   // idle events

cudaEvent_t take_event() {
  if (!g_evpool.empty()) {
    cudaEvent_t e = g_evpool.back();
    g_evpool.pop_back();
    return e;
  }
  cudaEvent_t e = nullptr;
  if (cudaEventCreate(&e) != cudaSuccess) return nullptr;
  return e;
}

// Enqueue one kernel through `launch`, counting it and, when tracing,
// bracketing it with events on the same stream.
template <class F>
pa_status run_launch(int32_t kind, const char* name, cudaStream_t stream, F&& launch) {
  cudaEvent_t b = nullptr, e = nullptr;
  {
    std::lock_guard<std::mutex> lk(g_trace_mu);
    if (g_trace_on && (int)g_trace.size() < kTraceCap) {
      b = take_event();
      e = take_event();
    }
  }
  if (b && e) cudaEventRecord(b, stream);
  const cudaError_t err = launch();
  if (b && e) {
    cudaEventRecord(e, stream);
    std::lock_guard<std::mutex> lk(g_trace_mu);
    g_trace.push_back({kind, b, e});
  }
  if (err != cudaSuccess) return fail(PA_ERR_CUDA, "%s: %s", name, cudaGetErrorString(err));
  g_launches.fetch_add(1, std::memory_order_relaxed);
  return PA_OK;
}

// --------------------------------------------------------------- planning
constexpr int kDecodeCtasPerSm = 3;  // resident decode CTAs per SM (shared memory bound)
constexpr int kSlotCap = 480;        // grid bound used for workspace sizing (>= SMs x 3)
constexpr int kMinSegPages = 8;      // fewest pages per CTA worth a CTA

int pages_of(int64_t len) { return (int)((len + pa::kPage - 1) / pa::kPage); }

// SM count of the current device, cached per device (atomics: host threads
// may race on a device's first call and store the same value).
int sm_count() {
  static std::atomic<int> cached[pa::kMaxDevices];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 148;
  const bool slot = dev >= 0 && dev < pa::kMaxDevices;
  if (slot) {
    const int c = cached[dev].load(std::memory_order_relaxed);
    if (c > 0) return c;
  }
  int n = 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 148;
  if (slot) cached[dev].store(n, std::memory_order_relaxed);
  return n;
}

// Largest persistent decode grid a call with these sizes may use (the
// workspace holds two partial slots per CTA).
int grid_cap(int32_t num_reqs, int32_t num_kv_heads, int32_t max_seq_len) {
  const int64_t rows = std::min<int64_t>(std::max(num_reqs, 0), pa::kPlanMaxRows);
  const int64_t items = rows * std::max(num_kv_heads, 1);
  const int64_t pages = items * std::max(1, pages_of(max_seq_len));
  // CTAs needed by the longest segments, rounded up to whole waves of kSlotCap
  int64_t g = (pages + pa::kDecodeMaxPagesPerCta - 1) / pa::kDecodeMaxPagesPerCta;
  g = std::max<int64_t>(1, (g + kSlotCap - 1) / kSlotCap) * kSlotCap;
  g = std::max<int64_t>(g, (items + 31) / 32);
  return (int)std::min<int64_t>(g, pa::kPlanMaxCtas);
}

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

// Workspace: [error word | item counters (num_reqs x Hkv int32) |
// partial o (2 x grid_cap x pieces_per_cta x 4 heads x D fp32) | partial lse
// (fp32)].  Sized for kDecodeWarps pieces per CTA of the CTA-granular grid
// bound: a CTA-granular CTA publishes fewer (one per CTA), a warp-granular
// launch (at most a third of the CTAs) one per warp segment (kWgWarps).
struct WorkspaceLayout {
  size_t counters, piece_o, piece_lse, total;
  int64_t slots;  // (piece, head) slots
};

WorkspaceLayout layout_for_grid(int32_t num_reqs, int32_t hkv, int32_t head_dim, int grid,
                                int pieces_per_cta = pa::kDecodeWarps) {
  WorkspaceLayout w;
  const size_t slots = (size_t)2 * grid * pieces_per_cta * PA_GQA_GROUP;
  w.slots = (int64_t)slots;
  w.counters = PA_ERROR_WORD_BYTES;
  w.piece_o = w.counters + align256((size_t)std::max(num_reqs, 0) * (size_t)hkv * 4);
  w.piece_lse = w.piece_o + align256(slots * (size_t)std::max(head_dim, 0) * 4);
  w.total = w.piece_lse + align256(slots * 4);
  return w;
}

WorkspaceLayout layout(int32_t num_reqs, int32_t num_q_heads, int32_t head_dim, int32_t max_seq_len) {
  const int32_t hkv = std::max(std::max(num_q_heads, 0) / PA_GQA_GROUP, 1);
  return layout_for_grid(num_reqs, hkv, head_dim, grid_cap(num_reqs, hkv, max_seq_len));
}

// Decode step: the launch shape, a function of the call's scalars only (so a
// captured launch is valid for every batch within them).  Segments per kv
// head: enough for one wave of resident CTAs when the largest stream allows
// it, and always enough that a segment of the largest stream holds at most
// kDecodeMaxPagesPerCta units.  -1 when that needs more than kPlanMaxCtas.
int step_grid(int32_t num_reqs, int32_t hkv, int32_t max_seq_len) {
  const int64_t cost = (int64_t)std::max(num_reqs, 0) * (pages_of(max_seq_len) + pa::kStepItemCost);
  const int64_t wave = std::max<int64_t>(1, (int64_t)sm_count() * kDecodeCtasPerSm / std::max(hkv, 1));
  int64_t nseg = std::min<int64_t>(wave, (cost + pa::kStepMinSegCost - 1) / pa::kStepMinSegCost);
  const int forced = g_forced_ctas.load();  // pa_set_decode_ctas
  if (forced > 0) nseg = (forced + std::max(hkv, 1) - 1) / std::max(hkv, 1);
  nseg = std::max<int64_t>(nseg, (cost + pa::kDecodeMaxPagesPerCta - 1) / pa::kDecodeMaxPagesPerCta);
  nseg = std::max<int64_t>(nseg, 1);
  if (nseg * hkv > pa::kPlanMaxCtas) return -1;
  return (int)(nseg * hkv);
}

// Decode step: whether a launch of nseg segments per kv head fits a kernel
// whose CTA holds at most max_items rows and max_pages pages of its segment
// in one window, for any lengths within the call's bounds.  A row costs at
// least 1 + kStepItemCost units and a segment is at most C units (C rounded
// up to a multiple of unit), C bounded by the largest total cost over the
// segments (or the minimum segment).
bool step_one_window(int32_t num_reqs, int64_t nseg, int32_t max_seq_len, int max_items, int max_pages, int unit) {
  const int64_t total_max = (int64_t)std::max(num_reqs, 0) * (pages_of(max_seq_len) + pa::kStepItemCost);
  const int64_t c_max =
      std::max<int64_t>(pa::kStepMinSegCost, (total_max + std::max<int64_t>(nseg, 1) - 1) / std::max<int64_t>(nseg, 1)) +
      unit;
  const bool items_fit = num_reqs + 1 <= max_items || c_max / (1 + pa::kStepItemCost) + 2 <= max_items;
  return items_fit && c_max <= max_pages;
}

// Shared-prefix pass: the chunk count for a call and the workspace region
// after the base layout: [prefix o (total_q x Hq x D fp32) | prefix lse |
// chunk o (chunks x total_q x Hq x D) | chunk lse | 2 x query tiles x Hkv
// int32 counters].  Chunks are sized so
// that chunks x Hkv x query tiles gives about one CTA per SM; kPrefixCtaCap
// bounds that for workspace sizing.
constexpr int kPrefixCtaCap = 512;
constexpr int kPrefixKeyTile = pa::kTcKeyTile;  // keys per tensor-core tile

int64_t prefix_qtiles(int32_t total_q) { return ((int64_t)std::max(total_q, 0) + pa::kPrefillQTile - 1) / pa::kPrefillQTile; }

int prefix_chunk_cap(int32_t total_q, int32_t hkv, int32_t prefix_pages) {
  const int64_t groups = std::max<int64_t>(1, prefix_qtiles(total_q) * std::max(hkv, 1));
  const int64_t tiles = ((int64_t)prefix_pages * pa::kPage + kPrefixKeyTile - 1) / kPrefixKeyTile;
  return (int)std::max<int64_t>(1, std::min<int64_t>(tiles, (kPrefixCtaCap + groups - 1) / groups));
}

struct PrefixLayout {
  size_t prefix_o, prefix_lse, chunk_o, chunk_lse, flags, total;
};

PrefixLayout prefix_layout(size_t base, int32_t total_q, int32_t num_q_heads, int32_t head_dim, int32_t prefix_pages) {
  PrefixLayout w;
  const int32_t hkv = std::max(std::max(num_q_heads, 0) / PA_GQA_GROUP, 1);
  const size_t rows = (size_t)std::max(total_q, 0) * (size_t)std::max(num_q_heads, 0);
  const int cap = prefix_chunk_cap(total_q, hkv, prefix_pages);
  const size_t chunk_rows = cap > 1 ? (size_t)cap * rows : 0;  // one chunk writes the prefix partial itself
  w.prefix_o = base;
  w.prefix_lse = w.prefix_o + align256(rows * (size_t)std::max(head_dim, 0) * 4);
  w.chunk_o = w.prefix_lse + align256(rows * 4);
  w.chunk_lse = w.chunk_o + align256(chunk_rows * (size_t)std::max(head_dim, 0) * 4);
  // per (query tile, kv head): chunks written, then folds done (a pass that
  // runs beside the decode launch); zero between calls
  w.flags = w.chunk_lse + align256(chunk_rows * 4);
  w.total = w.flags + align256((size_t)2 * prefix_qtiles(total_q) * hkv * 4);
  return w;
}

// Chunks of a shared-prefix pass that runs beside the decode launch, or 0
// when running it first is faster.  The pass takes chunks x groups SMs (one
// CTA each, groups = query tiles x kv heads) and the decode launch the other
// SMs; both should end together.  Rates measured on GB300: a prefix CTA
// takes ~1.05 us per 128-key tile after ~7 us of start-up and epilogue, and
// ~11 us as the first kernel of the step (128 CTAs starting at once); a
// decode SM streams ~46 GB/s after ~7 us of start-up and row ends.
// decode_slabs counts (page, kv head) slabs of 8 KiB.
int concurrent_prefix_chunks(int64_t key_tiles, int64_t groups, int64_t decode_slabs, int chunk_cap) {
  const int sms = sm_count();
  const double decode_bytes = (double)decode_slabs * 2 * pa::kSlabBytesHost;
  auto decode_us = [&](int64_t free_sms) { return 7.0 + decode_bytes / ((double)free_sms * 46e3); };
  const int64_t serial_chunks = std::min<int64_t>(chunk_cap, std::max<int64_t>(1, (sms + groups - 1) / groups));
  const double serial = 11.0 + (double)((key_tiles + serial_chunks - 1) / serial_chunks) * 1.05 + decode_us(sms);
  double best = serial;
  int best_chunks = 0;
  for (int ch = 1; ch <= chunk_cap && ch * groups <= sms / 2; ++ch) {
    const double prefix = 7.0 + (double)((key_tiles + ch - 1) / ch) * 1.05;
    const double t = std::max(prefix, decode_us(sms - ch * groups));
    if (t < best) {
      best = t;
      best_chunks = ch;
    }
  }
  return best_chunks;
}

// Chunked-prefill jobs of a batch with decode rows: how many CTAs run them
// beside the decode launch, which takes the other SMs (0: the jobs run first,
// one CTA per job, and the decode launch after them on every SM).  job_tiles
// holds each job's key tiles in the kernel's job order; CTA b of G takes job
// b of every round of G jobs, in reverse order on odd rounds.  Measured
// rates: a job takes ~5 us plus ~1 us per 128-key tile when it runs alone,
// ~1.3x that beside the decode stream (the two share the DRAM), after ~4 us
// of start; the decode launch streams ~54 GB/s per SM, at most ~6.5 TB/s,
// plus ~12 us of start and row ends.  Of the CTA counts within 1 us of the
// best the smallest is taken (the decode keeps the most SMs).  decode_slabs
// counts (page, kv head) slabs of 8 KiB.
int prefill_beside_ctas(const std::vector<int32_t>& job_tiles, int64_t decode_slabs, int sms) {
  const int64_t n = (int64_t)job_tiles.size();
  if (n == 0 || decode_slabs == 0) return 0;
  const double decode_bytes = (double)decode_slabs * 2 * pa::kSlabBytesHost;
  auto decode_us = [&](int64_t free_sms) { return 12.0 + decode_bytes / std::min((double)free_sms * 54e3, 6.5e6); };
  auto tiles_us = [&](int64_t G) {
    std::vector<double> t((size_t)G, 0.0);
    for (int64_t u = 0; u < n; ++u) {
      const int64_t rnd = u / G, b = (rnd & 1) ? G - 1 - u % G : u % G;
      t[(size_t)b] += 5.0 + 1.0 * job_tiles[(size_t)u];
    }
    return 4.0 + *std::max_element(t.begin(), t.end());
  };
  const double serial = tiles_us(std::min<int64_t>(n, sms)) + decode_us(sms);
  std::vector<double> beside(sms / 2 + 1, INFINITY);
  double best = INFINITY;
  for (int g = 1; g <= sms / 2 && g < n; ++g) {
    beside[g] = std::max(1.3 * tiles_us(g), decode_us(sms - g));
    best = std::min(best, beside[g]);
  }
  if (best >= serial - 2.0) return 0;  // a clear gain only
  for (int g = 1; g <= sms / 2; ++g)
    if (beside[g] <= best + 1.0) return g;
  return 0;
}

// Persistent CTAs for a batch of tile jobs alone, each job one query tile
// of a row that reads its keys once (verify rows): such a launch is bound by
// one CTA's stream (its copy, MMA and softmax chain: ~1.28 us per 128-key
// tile) and by HBM shared among the CTAs running (~0.0116 us per tile per
// CTA).  Over rounds of G jobs in the kernel's order, a round takes its
// longest job's tiles x max(1.28, CTAs in the round x 0.0116) us; the grid
// is the one with the shortest sum, among the smallest grids for 0 to 3 more
// rounds than one CTA per SM gives.  Verify batch (512 jobs of 17-18 tiles),
// G = 104 / 116 / 128 / 136 / 144 / 152: measured 115.3 / 121.1 / 106.6 /
// 108.3 / 109.9 / 114.1 us, modelled 115.2 / 119.7 / 106.6 / 108.0 / 113.0 /
// 118.0 us; the model picks 128.
int prefill_alone_ctas(const std::vector<int32_t>& job_tiles, int sms) {
  const int64_t n = (int64_t)job_tiles.size();
  if (n == 0) return 0;
  auto cost = [&](int64_t g) {
    double t = 0.0;
    for (int64_t r0 = 0; r0 < n; r0 += g) {
      const int64_t r1 = std::min(n, r0 + g);
      int32_t longest = 0;
      for (int64_t u = r0; u < r1; ++u) longest = std::max(longest, job_tiles[(size_t)u]);
      t += longest * std::max(1.28, (double)(r1 - r0) * 0.0116);
    }
    return t;
  };
  const int64_t k0 = (n + sms - 1) / sms;  // rounds with one CTA per SM
  int64_t best_g = std::min<int64_t>(n, sms);
  double best = cost(best_g);
  for (int64_t k = k0; k <= k0 + 3; ++k) {
    const int64_t g = (n + k - 1) / k;  // the smallest grid with k rounds
    if (g < 1 || g > sms) continue;
    const double c = cost(g);
    if (c < best) {
      best = c;
      best_g = g;
    }
  }
  return (int)best_g;
}

// Plan one persistent decode launch over decode rows rows[0..n): fills
// plan, returns the grid size (0 when there is nothing to do, -1 when no
// valid plan exists within the limits).  The grid is n_seg x Hkv CTAs.
int plan_decode(const int32_t* rows, int n, const int32_t* seq_lens_host, const int32_t* qo_indptr_host,
                int page_offset, int num_kv_heads, int gcap, int slots, int unit, int max_pages, int max_items,
                pa::DecodePlan& plan) {
  std::vector<int32_t> pages(n);
  int64_t total = 0;  // pages of one kv head's stream
  int32_t longest = 0;
  for (int d = 0; d < n; ++d) {
    pages[d] = pages_of(seq_lens_host[rows[d]]) - page_offset;
    total += pages[d];
    longest = std::max(longest, pages[d]);
  }
  if (total == 0) return 0;
  // A row cut into m pieces costs its last CTA a merge of m partials, so
  // when few rows leave CTAs to spare, segments get longer than
  // kMinSegPages: a row of R pages costs about seg + c R / seg, least at
  // seg ~ sqrt(R / 2) pages (measured: 8 for 128-page rows, 16 for 512).
  const int64_t min_seg = std::max<int64_t>(kMinSegPages, std::llround(std::sqrt(longest / 2.0)));
  const int seg_cap = std::min(gcap / num_kv_heads, pa::kPlanMaxCtas);  // segments per stream
  if (seg_cap < 1) return -1;
  const int forced = g_forced_ctas.load();
  int64_t nseg = forced > 0 ? (forced + num_kv_heads - 1) / num_kv_heads
                            : std::min<int64_t>(std::max(slots / num_kv_heads, 1), (total + min_seg - 1) / min_seg);
  nseg = std::max<int64_t>(1, std::min<int64_t>(nseg, seg_cap));
  // a segment holds at most max_pages pages; when that forces more segments
  // than one wave has slots, use whole waves so no wave runs part-empty
  const int64_t wave = std::max<int64_t>(1, slots / num_kv_heads);
  const int64_t need = (total + max_pages - 1) / max_pages;
  if (forced <= 0 && need > nseg) nseg = std::min<int64_t>((need + wave - 1) / wave * wave, seg_cap);
  int64_t seg = (total + nseg - 1) / nseg;
  seg = std::max<int64_t>(seg, (total + seg_cap - 1) / seg_cap);
  seg = (seg + unit - 1) / unit * unit;  // whole warp segments for the warp-granular kernel (unit kWgWarps)
  seg = std::min<int64_t>(seg, max_pages / unit * unit);  // more segments if one would be too long
  static_assert(pa::kWgMaxPagesPerCta % pa::kWgWarps == 0, "segments hold whole warp segments");
  for (;;) {
    const int ns = (int)((total + seg - 1) / seg);
    if (ns > seg_cap) return -1;
    // walk the row stream once: first row / page of every segment and the
    // most rows any segment touches
    int64_t d = 0, d_start = 0, max_items_seen = 0;
    for (int sidx = 0; sidx < ns; ++sidx) {
      const int64_t S = (int64_t)sidx * seg, E = std::min(total, S + seg);
      while (d_start + pages[d] <= S) d_start += pages[d++];
      plan.first_row[sidx] = (int32_t)d;
      plan.first_page[sidx] = (int32_t)(S - d_start);
      int64_t d2 = d, st2 = d_start, cnt = 0;
      while (d2 < n && st2 < E) {
        ++cnt;
        st2 += pages[d2++];
      }
      max_items_seen = std::max(max_items_seen, cnt);
    }
    if (max_items_seen <= max_items) {
      plan.n_rows = n;
      plan.seg = (int32_t)seg;
      plan.total = (int32_t)total;
      for (int r = 0; r < n; ++r) {
        plan.rows[r] = rows[r];
        plan.seq[r] = seq_lens_host[rows[r]];
        plan.tok[r] = qo_indptr_host[rows[r]];
      }
      return ns * num_kv_heads;
    }
    if (seg <= unit) return -1;
    // shorter segments touch fewer rows
    seg = ((seg + 1) / 2 + unit - 1) / unit * unit;
  }
}

// The decode launch over rows[0..n): segments of whole pages for the
// CTA-granular kernel; when they are long enough for four warp segments of
// kMinWarpSegPages (or a pass runs beside the launch, or the timeout
// diagnostic is on), planned again in whole warp segments for the
// warp-granular kernel, one CTA per SM (a third of the CTA-granular slots and
// grid bound, so the workspace's pieces cover its warps).  With no
// warp-granular plan within its limits, the CTA-granular kernel (beside
// prefill jobs too: it waits for them at its start, so they run first; beside
// a prefix pass it cannot run, as it does not fold the pass's chunks).
// Returns the grid (0: nothing to do, -1: no plan) and sets cta_granular.
int choose_decode_plan(const int32_t* rows, int n, const int32_t* seq_lens_host, const int32_t* qo_indptr_host,
                       int page_offset, int num_kv_heads, int gcap, int slots, bool concurrent, bool diag,
                       pa::DecodePlan& plan, bool& cta_granular) {
  auto plan_cta = [&] {
    return plan_decode(rows, n, seq_lens_host, qo_indptr_host, page_offset, num_kv_heads, gcap, slots, 1,
                       pa::kDecodeMaxPagesPerCta, pa::kDecodeMaxItemsPerCta, plan);
  };
  int grid = plan_cta();
  cta_granular = grid > 0 && !concurrent && !diag && plan.seg < pa::kDecodeWarps * pa::kMinWarpSegPages;
  static_assert(pa::kWgWarps <= kDecodeCtasPerSm * pa::kDecodeWarps, "warp-granular pieces fit the workspace");
  if (grid > 0 && !cta_granular) {
    grid = plan_decode(rows, n, seq_lens_host, qo_indptr_host, page_offset, num_kv_heads, gcap / kDecodeCtasPerSm,
                       slots / kDecodeCtasPerSm, pa::kWgWarps, pa::kWgMaxPagesPerCta, pa::kWgMaxItemsPerCta, plan);
    if (grid < 0 && (!concurrent || page_offset == 0) && !diag) {
      grid = plan_cta();
      cta_granular = grid > 0;
    }
  }
  return grid;
}

// ------------------------------------------------------------- TMA maps
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static const PFN_cuTensorMapEncodeTiled_v12000 fn = [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      f = nullptr;
    return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  }();
  return fn;
}

// Tiled maps of q ([total_q][Hq][128] bf16, boxes 64 x 4 heads x 32 tokens)
// and of the K / V pools (rows of 128 bf16, one per (block, kv head, token),
// boxes 64 x 16 rows), 128-byte swizzled; out-of-range q tokens read as 0.
pa_status make_tc_maps(const void* q, int32_t total_q, int32_t num_q_heads, const void* k_cache, const void* v_cache,
                       int64_t num_blocks, int32_t num_kv_heads, pa::TcMaps& m) {
  const PFN_cuTensorMapEncodeTiled_v12000 enc = encode_fn();
  if (!enc) return fail(PA_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
  const int64_t rows = num_blocks * num_kv_heads * pa::kPage;
  if (rows >= (int64_t(1) << 31)) return fail(PA_ERR_UNSUPPORTED, "pool of %lld rows: too many for the tile kernels",
                                               (long long)rows);
  const cuuint32_t estr[3] = {1, 1, 1};
  const cuuint64_t qdims[3] = {(cuuint64_t)pa::kHeadDim, (cuuint64_t)num_q_heads, (cuuint64_t)total_q};
  const cuuint64_t qstrides[2] = {(cuuint64_t)pa::kHeadDim * 2, (cuuint64_t)num_q_heads * pa::kHeadDim * 2};
  const cuuint32_t qbox[3] = {64, (cuuint32_t)pa::kGroup, (cuuint32_t)pa::kPrefillQTile};
  CUresult r = enc(&m.q, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(q), qdims, qstrides, qbox, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(PA_ERR_CUDA, "encoding the q tensor map: CUresult %d", (int)r);
  const cuuint64_t kdims[2] = {(cuuint64_t)pa::kHeadDim, (cuuint64_t)rows};
  const cuuint64_t kstrides[1] = {(cuuint64_t)pa::kHeadDim * 2};
  const cuuint32_t kbox[2] = {64, (cuuint32_t)pa::kPage};
  r = enc(&m.k, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(k_cache), kdims, kstrides, kbox, estr,
          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(PA_ERR_CUDA, "encoding the K tensor map: CUresult %d", (int)r);
  r = enc(&m.v, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(v_cache), kdims, kstrides, kbox, estr,
          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(PA_ERR_CUDA, "encoding the V tensor map: CUresult %d", (int)r);
  return PA_OK;
}

pa_status check_shape(int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim, int32_t block_size) {
  if (num_q_heads <= 0 || num_kv_heads <= 0 || head_dim <= 0 || block_size <= 0)
    return fail(PA_ERR_INVALID_ARG, "head counts, head_dim and block_size must be positive");
  if (head_dim != PA_HEAD_DIM) return fail(PA_ERR_UNSUPPORTED, "head_dim %d (only %d)", head_dim, PA_HEAD_DIM);
  if (block_size != PA_BLOCK_SIZE)
    return fail(PA_ERR_UNSUPPORTED, "block_size %d (only %d)", block_size, PA_BLOCK_SIZE);
  if (num_q_heads != PA_GQA_GROUP * num_kv_heads)
    return fail(PA_ERR_UNSUPPORTED, "num_q_heads %d != %d x num_kv_heads %d", num_q_heads, PA_GQA_GROUP,
                num_kv_heads);
  if (num_kv_heads > 256) return fail(PA_ERR_UNSUPPORTED, "num_kv_heads %d > 256", num_kv_heads);
  return PA_OK;
}

}  // namespace

pa_status pa::set_error(pa_status s, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_msg, sizeof g_msg, fmt, ap);
  va_end(ap);
  return s;
}

namespace {

// The attention entry points.  prefix_pages > 0: the first prefix_pages
// pages of every request are one shared prefix, attended once for all
// queries by the prefix pass and folded into each row's own part.  q8: the
// pools hold q8_0 pages (decode rows only).
pa_status attention(const void* q, const void* k_cache, const void* v_cache, int64_t num_blocks,
                    const int32_t* block_tables, int32_t max_blocks_per_req, const int32_t* seq_lens,
                    const int32_t* qo_indptr, const int32_t* seq_lens_host, const int32_t* qo_indptr_host,
                    int32_t num_reqs, int32_t total_q, int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                    int32_t block_size, int32_t prefix_pages, float sm_scale, void* out, float* lse, void* workspace,
                    size_t workspace_bytes, cudaStream_t stream, bool q8 = false) {
  pa_status s = check_shape(num_q_heads, num_kv_heads, head_dim, block_size);
  if (s != PA_OK) return s;
  if (num_reqs < 0 || num_reqs > 65535) return fail(PA_ERR_INVALID_ARG, "num_reqs %d outside [0, 65535]", num_reqs);
  if (total_q < 0) return fail(PA_ERR_INVALID_ARG, "total_q %d < 0", total_q);
  if (num_blocks <= 0) return fail(PA_ERR_INVALID_ARG, "num_blocks must be positive");
  if (!(fabsf(sm_scale) < INFINITY)) return fail(PA_ERR_INVALID_ARG, "sm_scale must be finite");
  if (!seq_lens_host || !qo_indptr_host) return fail(PA_ERR_INVALID_ARG, "host metadata pointers are required");
  if (!k_cache || !v_cache || !workspace || !seq_lens || !qo_indptr || (num_reqs > 0 && !block_tables) ||
      (total_q > 0 && (!q || !out)))
    return fail(PA_ERR_INVALID_ARG, "null device pointer");
  if (!aligned(q, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16) || !aligned(out, 16) ||
      !aligned(workspace, 256) || !aligned(lse, 4) || !aligned(block_tables, 4))
    return fail(PA_ERR_INVALID_ARG, "q, caches and out must be 16-byte aligned, workspace 256-byte aligned");
  if (qo_indptr_host[0] != 0) return fail(PA_ERR_INVALID_ARG, "qo_indptr[0] = %d, must be 0", qo_indptr_host[0]);
  if (qo_indptr_host[num_reqs] != total_q)
    return fail(PA_ERR_INVALID_ARG, "qo_indptr[num_reqs] = %d != total_q = %d", qo_indptr_host[num_reqs], total_q);

  if (prefix_pages < 0 || prefix_pages > max_blocks_per_req)
    return fail(PA_ERR_INVALID_ARG, "shared_prefix_pages %d outside [0, max_blocks_per_req %d]", prefix_pages,
                max_blocks_per_req);
  // classify rows and collect the plan inputs
  std::vector<int32_t> decode_rows;
  int32_t active = 0, first_active = -1;
  int32_t max_len = 1;
  std::vector<std::pair<int32_t, int32_t>> tiles;  // (kv extent of the tile, item index) for ordering
  static thread_local pa::PrefillItems items;
  std::vector<int32_t> item_req, item_q0;
  for (int r = 0; r < num_reqs; ++r) {
    const int32_t qo_len = qo_indptr_host[r + 1] - qo_indptr_host[r];
    const int32_t L = seq_lens_host[r];
    if (qo_len < 0) return fail(PA_ERR_INVALID_ARG, "qo_indptr decreases at request %d", r);
    if (L < 0 || L > PA_MAX_SEQ_LEN)
      return fail(L < 0 ? PA_ERR_INVALID_ARG : PA_ERR_UNSUPPORTED, "seq_lens[%d] = %d outside [0, %d]", r, L,
                  PA_MAX_SEQ_LEN);
    if (qo_len > L) return fail(PA_ERR_INVALID_ARG, "request %d: qo_len %d > seq_len %d", r, qo_len, L);
    if (pages_of(L) > max_blocks_per_req)
      return fail(PA_ERR_INVALID_ARG, "request %d: %d pages > max_blocks_per_req %d", r, pages_of(L),
                  max_blocks_per_req);
    max_len = std::max(max_len, L);
    if (q8 && qo_len > 1)
      return fail(PA_ERR_UNSUPPORTED, "request %d: q8_0 pages serve decode rows only (qo_len %d)", r, qo_len);
    if (qo_len > 0) {
      if (first_active < 0) first_active = r;
      ++active;
      if ((int64_t)L - qo_len < (int64_t)prefix_pages * pa::kPage)
        return fail(PA_ERR_INVALID_ARG, "request %d: the shared prefix (%d pages) must be cached before its %d queries",
                    r, prefix_pages, qo_len);
    }
    if (qo_len == 1) {
      decode_rows.push_back(r);
    } else if (qo_len > 1) {
      for (int32_t j0 = 0; j0 < qo_len; j0 += pa::kPrefillQTile) {
        tiles.push_back({L - qo_len + std::min(qo_len, j0 + pa::kPrefillQTile), (int32_t)item_req.size()});
        item_req.push_back(r);
        item_q0.push_back(j0);
      }
    }
  }
  const WorkspaceLayout wl = layout(num_reqs, num_q_heads, head_dim, max_len);
  const PrefixLayout pl = prefix_layout(wl.total, total_q, num_q_heads, head_dim, prefix_pages);
  const size_t need = prefix_pages > 0 ? pl.total : wl.total;
  if (workspace_bytes < need)
    return fail(PA_ERR_WORKSPACE_TOO_SMALL, "workspace %zu < %zu bytes", workspace_bytes, need);
  if (total_q == 0) return ok();
  // a prefix read by one request only is not worth a separate pass
  const int32_t P = active >= 2 ? prefix_pages : 0;
  if (P > 0 && prefix_qtiles(total_q) > 65535)
    return fail(PA_ERR_UNSUPPORTED, "total_q %d too large for the shared-prefix pass", total_q);

  char* ws = static_cast<char*>(workspace);
  int* err = reinterpret_cast<int*>(ws);
  const float scale_log2 = sm_scale * pa::kLog2e;
  float* prefix_o = P > 0 ? reinterpret_cast<float*>(ws + pl.prefix_o) : nullptr;
  float* prefix_lse = P > 0 ? reinterpret_cast<float*>(ws + pl.prefix_lse) : nullptr;
  static thread_local pa::TcMaps maps;
  if (P > 0 || !tiles.empty()) {
    s = make_tc_maps(q, total_q, num_q_heads, k_cache, v_cache, num_blocks, num_kv_heads, maps);
    if (s != PA_OK) return s;
  }

  // what the decode kernel folds in: the merged prefix partial, or the key-
  // chunk partials themselves when there is no prefill row to share them with
  const float* dec_prefix_o = prefix_o;
  const float* dec_prefix_lse = prefix_lse;
  int32_t dec_prefix_n = 1;
  // A decode-only batch (one decode launch, bf16 pages) may run the prefix
  // pass beside its decode launch: the pass on a few SMs, the decode CTAs on
  // the others, each row's fold waiting for its query tile's prefix chunks.
  const bool decode_only = P > 0 && tiles.empty() && !decode_rows.empty() && !q8 &&
                           decode_rows.size() <= (size_t)pa::kPlanMaxRows && g_forced_ctas.load() <= 0;
  int64_t decode_pages_all = 0;  // pages of every decode row's own part (one kv head)
  if (decode_only)
    for (int32_t r : decode_rows) decode_pages_all += pages_of(seq_lens_host[r]) - P;
  bool concurrent = false;
  int decode_slots = sm_count() * kDecodeCtasPerSm;
  if (P > 0) {
    pa::PrefixParams xp;
    xp.q = static_cast<const uint16_t*>(q);
    xp.k_cache = static_cast<const uint16_t*>(k_cache);
    xp.v_cache = static_cast<const uint16_t*>(v_cache);
    xp.num_blocks = num_blocks;
    xp.block_tables = block_tables;
    xp.max_blocks_per_req = max_blocks_per_req;
    xp.table_row = first_active;
    xp.total_q = total_q;
    xp.num_q_heads = num_q_heads;
    xp.num_kv_heads = num_kv_heads;
    xp.prefix_keys = P * pa::kPage;
    // about one CTA per SM over chunks x kv heads x query tiles
    const int64_t groups = prefix_qtiles(total_q) * num_kv_heads;
    const int chunk_cap = prefix_chunk_cap(total_q, num_kv_heads, P);
    int n_chunks = (int)std::min<int64_t>(chunk_cap, std::max<int64_t>(1, (sm_count() + groups - 1) / groups));
    const int64_t key_tiles = ((int64_t)xp.prefix_keys + kPrefixKeyTile - 1) / kPrefixKeyTile;
    if (decode_only) {
      // or beside the decode launch, when the pass is long enough to hide
      const int conc = concurrent_prefix_chunks(key_tiles, groups, decode_pages_all * num_kv_heads, chunk_cap);
      if (conc > 0) {
        n_chunks = conc;
        concurrent = true;
      }
    }
    xp.chunk_keys = (int32_t)((key_tiles + n_chunks - 1) / n_chunks * kPrefixKeyTile);
    n_chunks = (int)((xp.prefix_keys + xp.chunk_keys - 1) / xp.chunk_keys);
    if (concurrent) decode_slots = std::max(1, sm_count() - (int)(n_chunks * groups)) * kDecodeCtasPerSm;
    xp.done = concurrent ? reinterpret_cast<int*>(ws + pl.flags) : nullptr;
    xp.scale_log2 = scale_log2;
    xp.chunk_o = reinterpret_cast<float*>(ws + pl.chunk_o);
    xp.chunk_lse = reinterpret_cast<float*>(ws + pl.chunk_lse);
    xp.prefix_o = prefix_o;
    xp.prefix_lse = prefix_lse;
    xp.err = err;
    s = run_launch(PA_KERNEL_PREFIX, "prefix", stream, [&] { return pa::launch_prefix(xp, n_chunks, maps, stream); });
    if (s != PA_OK) return s;
    if (n_chunks > 1 && tiles.empty()) {
      // decode rows only: the decode kernel folds the chunk partials itself
      dec_prefix_o = xp.chunk_o;
      dec_prefix_lse = xp.chunk_lse;
      dec_prefix_n = n_chunks;
    } else if (n_chunks > 1) {
      s = run_launch(PA_KERNEL_PREFIX_MERGE, "prefix_merge", stream,
                     [&] { return pa::launch_prefix_merge(xp, n_chunks, stream); });
      if (s != PA_OK) return s;
    }
  }

  int prefill_ctas = 0;  // CTAs of the prefill launch (0: one per job)
  if (!tiles.empty()) {
    // longest key extent first, so the big tiles do not form the tail
    std::stable_sort(tiles.begin(), tiles.end(), [](const auto& a, const auto& b) { return a.first > b.first; });
    // The jobs beside the decode launch (decode rows of bf16 pages, no shared
    // prefix, one launch of each): the tiles on a few SMs, the decode stream
    // on the others.
    const int forced_p = g_prefill_ctas.load();
    if (P == 0 && !q8 && !decode_rows.empty() && decode_rows.size() <= (size_t)pa::kPlanMaxRows &&
        tiles.size() <= (size_t)pa::kMaxPrefillItems && g_forced_ctas.load() <= 0 && g_decode_fault.load() == 0 &&
        forced_p >= 0) {
      const int jobs = (int)tiles.size() * num_kv_heads;
      if (forced_p > 0) {
        prefill_ctas = std::min(forced_p, std::min(jobs - 1, sm_count() / 2));
      } else {
        std::vector<int32_t> job_tiles;
        job_tiles.reserve((size_t)jobs);
        for (int h = 0; h < num_kv_heads; ++h)  // the kernel's job order when it runs several per CTA
          for (const auto& t : tiles) job_tiles.push_back((t.first + pa::kTcKeyTile - 1) / pa::kTcKeyTile);
        int64_t decode_pages = 0;
        for (int32_t r : decode_rows) decode_pages += pages_of(seq_lens_host[r]);
        prefill_ctas = prefill_beside_ctas(job_tiles, decode_pages * num_kv_heads, sm_count());
      }
      if (prefill_ctas > 0) {
        concurrent = true;
        decode_slots = std::max(1, sm_count() - prefill_ctas) * kDecodeCtasPerSm;
      }
    } else if (P == 0 && decode_rows.empty() && forced_p >= 0 && !q8 &&
               tiles.size() <= (size_t)pa::kMaxPrefillItems && g_forced_ctas.load() <= 0 &&
               g_decode_fault.load() == 0) {
      // a batch of tile jobs alone: persistent CTAs, each running its jobs
      // in turn with the next one's start overlapping this one's end, when
      // forced, or when every row is one query tile (verify rows) and there
      // are at least two jobs per SM, on the grid prefill_alone_ctas picks
      // (verify: one CTA per job 118.3 us, 152 persistent CTAs 116.3, 128
      // 110.0); chunks of longer prompts keep one CTA per job
      const int jobs = (int)tiles.size() * num_kv_heads;
      bool single_tiles = true;
      for (const auto& t : tiles) single_tiles = single_tiles && item_q0[(size_t)t.second] == 0 &&
                                               qo_indptr_host[item_req[(size_t)t.second] + 1] -
                                                       qo_indptr_host[item_req[(size_t)t.second]] <=
                                                   pa::kPrefillQTile;
      if (forced_p > 0) {
        prefill_ctas = std::min(forced_p, jobs - 1);
      } else if (single_tiles && jobs >= 2 * sm_count()) {
        std::vector<int32_t> job_tiles;
        job_tiles.reserve((size_t)jobs);
        for (int h = 0; h < num_kv_heads; ++h)  // the kernel's job order
          for (const auto& t : tiles) job_tiles.push_back((t.first + pa::kTcKeyTile - 1) / pa::kTcKeyTile);
        prefill_ctas = std::min(prefill_alone_ctas(job_tiles, sm_count()), jobs - 1);
      }
    }
    pa::PrefillParams pp;
    pp.q = static_cast<const uint16_t*>(q);
    pp.k_cache = static_cast<const uint16_t*>(k_cache);
    pp.v_cache = static_cast<const uint16_t*>(v_cache);
    pp.num_blocks = num_blocks;
    pp.block_tables = block_tables;
    pp.max_blocks_per_req = max_blocks_per_req;
    pp.seq_lens = seq_lens;
    pp.qo_indptr = qo_indptr;
    pp.num_q_heads = num_q_heads;
    pp.num_kv_heads = num_kv_heads;
    pp.scale_log2 = scale_log2;
    pp.kv_key_offset = P * pa::kPage;
    pp.prefix_o = prefix_o;
    pp.prefix_lse = prefix_lse;
    pp.out = static_cast<uint16_t*>(out);
    pp.lse = lse;
    pp.err = err;
    for (size_t base = 0; base < tiles.size(); base += pa::kMaxPrefillItems) {
      const size_t n = std::min(tiles.size() - base, (size_t)pa::kMaxPrefillItems);
      items.count = (int32_t)n;
      for (size_t i = 0; i < n; ++i) {
        const int32_t idx = tiles[base + i].second;
        items.req[i] = item_req[idx];
        items.q_start[i] = item_q0[idx];
      }
      s = run_launch(PA_KERNEL_PREFILL, "prefill", stream,
                     [&] { return pa::launch_prefill(pp, items, maps, prefill_ctas, stream); });
      if (s != PA_OK) return s;
    }
  }

  if (!decode_rows.empty()) {
    pa::DecodeParams dp{};
    dp.q = static_cast<const uint16_t*>(q);
    dp.k_cache = static_cast<const uint16_t*>(k_cache);
    dp.v_cache = static_cast<const uint16_t*>(v_cache);
    dp.num_blocks = num_blocks;
    dp.block_tables = block_tables;
    dp.max_blocks_per_req = max_blocks_per_req;
    dp.seq_lens = seq_lens;
    dp.qo_indptr = qo_indptr;
    dp.num_q_heads = num_q_heads;
    dp.num_kv_heads = num_kv_heads;
    dp.scale_log2 = scale_log2;
    dp.page_offset = P;
    dp.prefix_o = dec_prefix_o;
    dp.prefix_lse = dec_prefix_lse;
    dp.prefix_n = dec_prefix_n;
    dp.prefix_rows = (int64_t)total_q * num_q_heads;
    dp.prefix_done = concurrent && P > 0 ? reinterpret_cast<int*>(ws + pl.flags) : nullptr;
    dp.prefix_readers = concurrent && P > 0
                            ? reinterpret_cast<int*>(ws + pl.flags) + prefix_qtiles(total_q) * num_kv_heads
                            : nullptr;
    dp.beside = concurrent ? 1 : 0;
    dp.total_q = total_q;
    dp.out = static_cast<uint16_t*>(out);
    dp.lse = lse;
    dp.piece_o = reinterpret_cast<float*>(ws + wl.piece_o);
    dp.piece_lse = reinterpret_cast<float*>(ws + wl.piece_lse);
    dp.piece_slots = wl.slots;
    dp.counters = reinterpret_cast<int*>(ws + wl.counters);
    dp.err = err;
    static thread_local pa::DecodePlan plan;
    const int gcap = grid_cap(num_reqs, num_kv_heads, max_len);
    // one launch per kPlanMaxRows decode rows (the plan travels as kernel
    // parameters); launches on one stream run in order and reuse the slots
    for (size_t d0 = 0; d0 < decode_rows.size(); d0 += pa::kPlanMaxRows) {
      const int n = (int)std::min(decode_rows.size() - d0, (size_t)pa::kPlanMaxRows);
      // after a prefix pass that ends before it, or after the prefill tiles,
      // the decode CTAs go in plain stream order: resident early, waiting on
      // the tile kernel's tail, they made the step 1-2 us longer, not shorter.
      // Beside a concurrent prefix pass they start as soon as it has.
      const bool overlap = d0 > 0 || (P == 0 && tiles.empty()) || concurrent;
      const bool diag = !q8 && g_decode_fault.load() != 0;
      bool cta_granular = false;
      const int grid = choose_decode_plan(decode_rows.data() + d0, n, seq_lens_host, qo_indptr_host, P, num_kv_heads,
                                          gcap, decode_slots, concurrent, diag, plan, cta_granular);
      if (grid < 0) return fail(PA_ERR_UNSUPPORTED, "no decode plan within the kernel limits");
      if (grid == 0) continue;
      s = run_launch(PA_KERNEL_DECODE, "decode", stream,
                     [&] { return pa::launch_decode(dp, plan, grid, q8, overlap, diag, cta_granular, stream); });
      if (s != PA_OK) return s;
    }
  }
  return ok();
}

pa_status append(const void* k_new, const void* v_new, const int64_t* slot_mapping, int64_t n_tokens, void* k_cache,
                 void* v_cache, int64_t num_blocks, int32_t block_size, int32_t num_kv_heads, int32_t head_dim,
                 void* workspace, size_t workspace_bytes, pa_stream_t stream, bool q8);

}  // namespace

extern "C" {

int32_t pa_abi_version(void) { return PA_ABI_VERSION; }

const char* pa_status_string(int32_t s) {
  switch (s) {
    case PA_OK: return "PA_OK";
    case PA_ERR_INVALID_ARG: return "PA_ERR_INVALID_ARG";
    case PA_ERR_UNSUPPORTED: return "PA_ERR_UNSUPPORTED";
    case PA_ERR_WORKSPACE_TOO_SMALL: return "PA_ERR_WORKSPACE_TOO_SMALL";
    case PA_ERR_CUDA: return "PA_ERR_CUDA";
    case PA_ERR_DEVICE_INDEX: return "PA_ERR_DEVICE_INDEX";
    case PA_ERR_DEVICE_TIMEOUT: return "PA_ERR_DEVICE_TIMEOUT";
    default: return "PA_ERR_UNKNOWN";
  }
}

const char* pa_last_error_message(void) { return g_msg; }

pa_status pa_kv_append(const void* k_new, const void* v_new, const int64_t* slot_mapping, int64_t n_tokens,
                       void* k_cache, void* v_cache, int64_t num_blocks, int32_t block_size, int32_t num_kv_heads,
                       int32_t head_dim, void* workspace, size_t workspace_bytes, pa_stream_t stream) {
  return append(k_new, v_new, slot_mapping, n_tokens, k_cache, v_cache, num_blocks, block_size, num_kv_heads,
                head_dim, workspace, workspace_bytes, stream, false);
}

pa_status pa_kv_append_q8(const void* k_new, const void* v_new, const int64_t* slot_mapping, int64_t n_tokens,
                          void* k_cache, void* v_cache, int64_t num_blocks, int32_t block_size, int32_t num_kv_heads,
                          int32_t head_dim, void* workspace, size_t workspace_bytes, pa_stream_t stream) {
  return append(k_new, v_new, slot_mapping, n_tokens, k_cache, v_cache, num_blocks, block_size, num_kv_heads,
                head_dim, workspace, workspace_bytes, stream, true);
}

pa_status pa_attention_varlen_q8(const void* q, const void* k_cache, const void* v_cache, int64_t num_blocks,
                                 const int32_t* block_tables, int32_t max_blocks_per_req, const int32_t* seq_lens,
                                 const int32_t* qo_indptr, const int32_t* seq_lens_host,
                                 const int32_t* qo_indptr_host, int32_t num_reqs, int32_t total_q,
                                 int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim, int32_t block_size,
                                 float sm_scale, void* out, float* lse, void* workspace, size_t workspace_bytes,
                                 pa_stream_t stream) {
  return attention(q, k_cache, v_cache, num_blocks, block_tables, max_blocks_per_req, seq_lens, qo_indptr,
                   seq_lens_host, qo_indptr_host, num_reqs, total_q, num_q_heads, num_kv_heads, head_dim, block_size,
                   0, sm_scale, out, lse, workspace, workspace_bytes, stream, true);
}

}  // extern "C"

namespace {

pa_status append(const void* k_new, const void* v_new, const int64_t* slot_mapping, int64_t n_tokens, void* k_cache,
                 void* v_cache, int64_t num_blocks, int32_t block_size, int32_t num_kv_heads, int32_t head_dim,
                 void* workspace, size_t workspace_bytes, pa_stream_t stream, bool q8) {
  if (n_tokens < 0) return fail(PA_ERR_INVALID_ARG, "n_tokens %lld < 0", (long long)n_tokens);
  if (num_blocks <= 0) return fail(PA_ERR_INVALID_ARG, "num_blocks must be positive");
  pa_status s = check_shape(PA_GQA_GROUP * num_kv_heads, num_kv_heads, head_dim, block_size);
  if (s != PA_OK) return s;
  if (!k_cache || !v_cache || !workspace) return fail(PA_ERR_INVALID_ARG, "null cache or workspace pointer");
  if (n_tokens > 0 && (!k_new || !v_new || !slot_mapping)) return fail(PA_ERR_INVALID_ARG, "null input pointer");
  if (!aligned(k_new, 16) || !aligned(v_new, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16) ||
      !aligned(slot_mapping, 8) || !aligned(workspace, 4))
    return fail(PA_ERR_INVALID_ARG, "tensors must be 16-byte aligned (slot_mapping 8, workspace 4)");
  if (workspace_bytes < PA_ERROR_WORD_BYTES)
    return fail(PA_ERR_WORKSPACE_TOO_SMALL, "workspace %zu < %d bytes", workspace_bytes, PA_ERROR_WORD_BYTES);
  if (n_tokens == 0) return ok();
  pa::AppendParams p;
  p.k_new = static_cast<const uint16_t*>(k_new);
  p.v_new = static_cast<const uint16_t*>(v_new);
  p.slot_mapping = slot_mapping;
  p.n_tokens = n_tokens;
  p.k_cache = static_cast<uint16_t*>(k_cache);
  p.v_cache = static_cast<uint16_t*>(v_cache);
  p.num_blocks = num_blocks;
  p.num_kv_heads = num_kv_heads;
  p.err = static_cast<int*>(workspace);
  s = run_launch(PA_KERNEL_KV_APPEND, q8 ? "kv_append_q8" : "kv_append", stream,
                 [&] { return q8 ? pa::launch_kv_append_q8(p, stream) : pa::launch_kv_append(p, stream); });
  return s == PA_OK ? ok() : s;
}

}  // namespace

extern "C" {

pa_status pa_copy_blocks(const int32_t* src_blocks, const int32_t* dst_blocks, int64_t n_pairs, void* k_cache,
                         void* v_cache, int64_t num_blocks, int32_t block_size, int32_t num_kv_heads,
                         int32_t head_dim, void* workspace, size_t workspace_bytes, pa_stream_t stream) {
  if (n_pairs < 0) return fail(PA_ERR_INVALID_ARG, "n_pairs %lld < 0", (long long)n_pairs);
  if (num_blocks <= 0) return fail(PA_ERR_INVALID_ARG, "num_blocks must be positive");
  pa_status s = check_shape(PA_GQA_GROUP * num_kv_heads, num_kv_heads, head_dim, block_size);
  if (s != PA_OK) return s;
  if (!k_cache || !v_cache || !workspace) return fail(PA_ERR_INVALID_ARG, "null cache or workspace pointer");
  if (n_pairs > 0 && (!src_blocks || !dst_blocks)) return fail(PA_ERR_INVALID_ARG, "null block id pointer");
  if (!aligned(k_cache, 16) || !aligned(v_cache, 16) || !aligned(src_blocks, 4) || !aligned(dst_blocks, 4) ||
      !aligned(workspace, 4))
    return fail(PA_ERR_INVALID_ARG, "caches must be 16-byte aligned (block ids and workspace 4)");
  if (workspace_bytes < PA_ERROR_WORD_BYTES)
    return fail(PA_ERR_WORKSPACE_TOO_SMALL, "workspace %zu < %d bytes", workspace_bytes, PA_ERROR_WORD_BYTES);
  if (n_pairs == 0) return ok();
  pa::CopyParams p;
  p.k_cache = static_cast<uint16_t*>(k_cache);
  p.v_cache = static_cast<uint16_t*>(v_cache);
  p.num_blocks = num_blocks;
  p.src = src_blocks;
  p.dst = dst_blocks;
  p.n_pairs = n_pairs;
  p.block_vecs = (int64_t)num_kv_heads * block_size * head_dim * 2 / 16;
  p.err = static_cast<int*>(workspace);
  s = run_launch(PA_KERNEL_COPY_BLOCKS, "copy_blocks", stream, [&] { return pa::launch_copy_blocks(p, stream); });
  return s == PA_OK ? ok() : s;
}

size_t pa_attention_workspace_size(int32_t num_reqs, int32_t total_q, int32_t num_q_heads, int32_t head_dim,
                                   int32_t max_seq_len) {
  if (num_reqs < 0 || total_q < 0 || num_q_heads < 0 || head_dim < 0) return 0;
  return layout(num_reqs, num_q_heads, head_dim, std::max(max_seq_len, 1)).total;
}

pa_status pa_attention_varlen(const void* q, const void* k_cache, const void* v_cache, int64_t num_blocks,
                              const int32_t* block_tables, int32_t max_blocks_per_req, const int32_t* seq_lens,
                              const int32_t* qo_indptr, const int32_t* seq_lens_host, const int32_t* qo_indptr_host,
                              int32_t num_reqs, int32_t total_q, int32_t num_q_heads, int32_t num_kv_heads,
                              int32_t head_dim, int32_t block_size, float sm_scale, void* out, float* lse,
                              void* workspace, size_t workspace_bytes, pa_stream_t stream) {
  return attention(q, k_cache, v_cache, num_blocks, block_tables, max_blocks_per_req, seq_lens, qo_indptr,
                   seq_lens_host, qo_indptr_host, num_reqs, total_q, num_q_heads, num_kv_heads, head_dim, block_size,
                   0, sm_scale, out, lse, workspace, workspace_bytes, stream);
}

size_t pa_decode_step_workspace_size(int32_t num_reqs, int32_t num_q_heads, int32_t head_dim,
                                     int32_t max_seq_len) {
  if (num_reqs < 0 || num_reqs > pa::kPlanMaxRows || num_q_heads < PA_GQA_GROUP || head_dim < 0 || max_seq_len < 1 ||
      max_seq_len > PA_MAX_SEQ_LEN)
    return 0;
  const int32_t hkv = num_q_heads / PA_GQA_GROUP;
  const int grid = step_grid(num_reqs, hkv, max_seq_len);
  if (grid < 0) return 0;
  return layout_for_grid(num_reqs, hkv, head_dim, grid).total;
}

int32_t pa_decode_step_bucket(int32_t num_reqs) {
  if (num_reqs < 0 || num_reqs > pa::kPlanMaxRows) return -1;
  int32_t b = 1;
  while (b < num_reqs) b <<= 1;
  return b;
}

pa_status pa_decode_step(const void* q, const void* k_new, const void* v_new, void* k_cache, void* v_cache,
                         int64_t num_blocks, const int32_t* block_tables, int32_t max_blocks_per_req,
                         const int32_t* seq_lens, int32_t num_reqs, int32_t max_seq_len, int32_t num_q_heads,
                         int32_t num_kv_heads, int32_t head_dim, int32_t block_size, float sm_scale, void* out,
                         float* lse, void* workspace, size_t workspace_bytes, pa_stream_t stream) {
  pa_status s = check_shape(num_q_heads, num_kv_heads, head_dim, block_size);
  if (s != PA_OK) return s;
  if (num_reqs < 0 || num_reqs > pa::kPlanMaxRows)
    return fail(PA_ERR_UNSUPPORTED, "num_reqs %d outside [0, %d]", num_reqs, pa::kPlanMaxRows);
  if (max_seq_len < 1 || max_seq_len > PA_MAX_SEQ_LEN)
    return fail(PA_ERR_INVALID_ARG, "max_seq_len %d outside [1, %d]", max_seq_len, PA_MAX_SEQ_LEN);
  if (num_blocks <= 0) return fail(PA_ERR_INVALID_ARG, "num_blocks must be positive");
  if (max_blocks_per_req < 1) return fail(PA_ERR_INVALID_ARG, "max_blocks_per_req must be positive");
  if (!(fabsf(sm_scale) < INFINITY)) return fail(PA_ERR_INVALID_ARG, "sm_scale must be finite");
  if (!workspace || !k_cache || !v_cache ||
      (num_reqs > 0 && (!q || !k_new || !v_new || !block_tables || !seq_lens || !out)))
    return fail(PA_ERR_INVALID_ARG, "null device pointer");
  if (!aligned(q, 16) || !aligned(k_new, 16) || !aligned(v_new, 16) || !aligned(k_cache, 16) ||
      !aligned(v_cache, 16) || !aligned(out, 16) || !aligned(workspace, 256) || !aligned(lse, 4) ||
      !aligned(block_tables, 4) || !aligned(seq_lens, 4))
    return fail(PA_ERR_INVALID_ARG, "q, k_new, v_new, caches and out must be 16-byte aligned, workspace 256-byte aligned");
  const int grid = step_grid(num_reqs, num_kv_heads, max_seq_len);
  if (grid < 0)
    return fail(PA_ERR_UNSUPPORTED, "%d rows of up to %d tokens need more than %d CTAs", num_reqs, max_seq_len,
                pa::kPlanMaxCtas);
  const WorkspaceLayout wl = layout_for_grid(num_reqs, num_kv_heads, head_dim, grid);
  if (workspace_bytes < wl.total)
    return fail(PA_ERR_WORKSPACE_TOO_SMALL, "workspace %zu < %zu bytes", workspace_bytes, wl.total);
  if (num_reqs == 0) return ok();

  char* ws = static_cast<char*>(workspace);
  pa::DecodeParams dp{};
  dp.q = static_cast<const uint16_t*>(q);
  dp.k_cache = static_cast<const uint16_t*>(k_cache);
  dp.v_cache = static_cast<const uint16_t*>(v_cache);
  dp.num_blocks = num_blocks;
  dp.block_tables = block_tables;
  dp.max_blocks_per_req = max_blocks_per_req;
  dp.seq_lens = seq_lens;
  dp.num_q_heads = num_q_heads;
  dp.num_kv_heads = num_kv_heads;
  dp.scale_log2 = sm_scale * pa::kLog2e;
  dp.out = static_cast<uint16_t*>(out);
  dp.lse = lse;
  dp.piece_o = reinterpret_cast<float*>(ws + wl.piece_o);
  dp.piece_lse = reinterpret_cast<float*>(ws + wl.piece_lse);
  dp.piece_slots = wl.slots;
  dp.counters = reinterpret_cast<int*>(ws + wl.counters);
  dp.err = reinterpret_cast<int*>(ws);
  dp.k_new = static_cast<const uint16_t*>(k_new);
  dp.v_new = static_cast<const uint16_t*>(v_new);
  dp.k_store = static_cast<uint16_t*>(k_cache);
  dp.v_store = static_cast<uint16_t*>(v_cache);
  pa::StepPlan plan;
  plan.n_rows = num_reqs;
  plan.max_seq_len = max_seq_len;
  // the warp-granular kernel (one CTA per SM: a third of the segments, so
  // that its kWgWarps pieces per CTA fit the workspace's kDecodeWarps per
  // CTA-granular CTA) when its segments fit one window and the CTA-granular
  // segments the bounds allow hold four warp segments of kMinWarpSegPages
  // (the same rule as the host plan's; from the bounds, so a captured launch
  // keeps its kernel)
  const int64_t nseg = std::max(1, grid / num_kv_heads);
  const int64_t nseg_wg = nseg / kDecodeCtasPerSm;
  static_assert(pa::kWgWarps <= kDecodeCtasPerSm * pa::kDecodeWarps, "warp-granular pieces fit the workspace");
  const int64_t seg_est = ((int64_t)num_reqs * (pages_of(max_seq_len) + pa::kStepItemCost) + nseg - 1) / nseg;
  const bool warp_granular =
      nseg_wg >= 1 &&
      step_one_window(num_reqs, nseg_wg, max_seq_len, pa::kWgMaxItemsPerCta, pa::kWgMaxPagesPerCta, pa::kWgWarps) &&
      seg_est >= pa::kDecodeWarps * pa::kMinWarpSegPages;
  const int launch_grid = warp_granular ? (int)(nseg_wg * num_kv_heads) : grid;
  s = run_launch(PA_KERNEL_DECODE_STEP, "decode_step", stream,
                 [&] { return pa::launch_decode_step(dp, plan, launch_grid, warp_granular, stream); });
  return s == PA_OK ? ok() : s;
}

size_t pa_shared_prefix_workspace_size(int32_t num_reqs, int32_t total_q, int32_t num_q_heads, int32_t head_dim,
                                       int32_t max_seq_len, int32_t shared_prefix_pages) {
  if (num_reqs < 0 || total_q < 0 || num_q_heads < 0 || head_dim < 0 || shared_prefix_pages < 0) return 0;
  const size_t base = layout(num_reqs, num_q_heads, head_dim, std::max(max_seq_len, 1)).total;
  if (shared_prefix_pages == 0) return base;
  return prefix_layout(base, total_q, num_q_heads, head_dim, shared_prefix_pages).total;
}

pa_status pa_attention_varlen_shared_prefix(
    const void* q, const void* k_cache, const void* v_cache, int64_t num_blocks, const int32_t* block_tables,
    int32_t max_blocks_per_req, const int32_t* seq_lens, const int32_t* qo_indptr, const int32_t* seq_lens_host,
    const int32_t* qo_indptr_host, int32_t num_reqs, int32_t total_q, int32_t num_q_heads, int32_t num_kv_heads,
    int32_t head_dim, int32_t block_size, int32_t shared_prefix_pages, float sm_scale, void* out, float* lse,
    void* workspace, size_t workspace_bytes, pa_stream_t stream) {
  return attention(q, k_cache, v_cache, num_blocks, block_tables, max_blocks_per_req, seq_lens, qo_indptr,
                   seq_lens_host, qo_indptr_host, num_reqs, total_q, num_q_heads, num_kv_heads, head_dim, block_size,
                   shared_prefix_pages, sm_scale, out, lse, workspace, workspace_bytes, stream);
}

pa_status pa_merge_lse(const void* o_a, const float* lse_a, const void* o_b, const float* lse_b, void* o_out,
                       float* lse_out, int64_t rows, int32_t num_heads, int32_t head_dim, pa_stream_t stream) {
  if (rows < 0 || num_heads <= 0 || head_dim <= 0 || head_dim % 8 != 0)
    return fail(PA_ERR_INVALID_ARG, "rows >= 0, num_heads > 0 and head_dim a positive multiple of 8 required");
  if (rows == 0) return ok();
  if (!o_a || !lse_a || !o_b || !lse_b || !o_out) return fail(PA_ERR_INVALID_ARG, "null pointer");
  if (!aligned(o_a, 16) || !aligned(o_b, 16) || !aligned(o_out, 16))
    return fail(PA_ERR_INVALID_ARG, "o tensors must be 16-byte aligned");
  if (lse_out) {
    const size_t n = (size_t)rows * num_heads * sizeof(float);
    auto overlap = [n](const void* a, const void* b) {
      const char* x = static_cast<const char*>(a);
      const char* y = static_cast<const char*>(b);
      return x < y + n && y < x + n;
    };
    if (overlap(lse_out, lse_a) || overlap(lse_out, lse_b))
      return fail(PA_ERR_INVALID_ARG, "lse_out must not overlap lse_a or lse_b");
  }
  pa::MergeParams p;
  p.o_a = static_cast<const uint16_t*>(o_a);
  p.lse_a = lse_a;
  p.o_b = static_cast<const uint16_t*>(o_b);
  p.lse_b = lse_b;
  p.o_out = static_cast<uint16_t*>(o_out);
  p.lse_out = lse_out;
  p.rows = rows;
  p.num_heads = num_heads;
  p.head_dim = head_dim;
  pa_status s = run_launch(PA_KERNEL_MERGE, "merge_lse", stream, [&] { return pa::launch_merge(p, stream); });
  return s == PA_OK ? ok() : s;
}

pa_status pa_get_device_error(const void* workspace, int32_t* code_out) {
  if (!workspace || !code_out) return fail(PA_ERR_INVALID_ARG, "null pointer");
  int32_t v = 0;
  const cudaError_t e = cudaMemcpy(&v, workspace, sizeof v, cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return fail(PA_ERR_CUDA, "reading the error word: %s", cudaGetErrorString(e));
  *code_out = v;
  return ok();
}

pa_status pa_clear_device_error(void* workspace, pa_stream_t stream) {
  if (!workspace) return fail(PA_ERR_INVALID_ARG, "null workspace");
  const cudaError_t e = cudaMemsetAsync(workspace, 0, sizeof(int32_t), stream);
  if (e != cudaSuccess) return fail(PA_ERR_CUDA, "clearing the error word: %s", cudaGetErrorString(e));
  return ok();
}

pa_status pa_set_decode_ctas(int32_t n) {
  if (n < 0 || n > pa::kPlanMaxCtas)
    return fail(PA_ERR_INVALID_ARG, "decode grid %d outside [0, %d]", n, pa::kPlanMaxCtas);
  g_forced_ctas.store(n);
  return ok();
}

pa_status pa_set_prefill_ctas(int32_t n) {
  if (n < -1 || n > pa::kPlanMaxCtas)
    return fail(PA_ERR_INVALID_ARG, "prefill CTAs %d outside [-1, %d]", n, pa::kPlanMaxCtas);
  g_prefill_ctas.store(n);
  return ok();
}

pa_status pa_plan_tile_grid(const int32_t* job_tiles, int32_t n_jobs, int64_t decode_slabs, int32_t sms,
                            int32_t* ctas) {
  if (!ctas) return fail(PA_ERR_INVALID_ARG, "ctas is null");
  *ctas = 0;
  if (n_jobs < 0 || n_jobs > pa::kMaxPrefillItems * 256 || (n_jobs > 0 && !job_tiles))
    return fail(PA_ERR_INVALID_ARG, "job_tiles must hold n_jobs = %d counts (at most %d)", n_jobs,
                pa::kMaxPrefillItems * 256);
  if (sms < 1 || sms > pa::kPlanMaxCtas) return fail(PA_ERR_INVALID_ARG, "sms %d outside [1, %d]", sms, pa::kPlanMaxCtas);
  if (decode_slabs < 0) return fail(PA_ERR_INVALID_ARG, "decode_slabs %lld < 0", (long long)decode_slabs);
  std::vector<int32_t> tiles(job_tiles, job_tiles + n_jobs);
  for (int32_t i = 0; i < n_jobs; ++i)
    if (tiles[(size_t)i] < 1) return fail(PA_ERR_INVALID_ARG, "job %d has %d key tiles (>= 1)", i, tiles[(size_t)i]);
  if (n_jobs == 0) return ok();
  if (decode_slabs > 0)
    *ctas = prefill_beside_ctas(tiles, decode_slabs, sms);  // (fewer than the jobs, at most half the SMs)
  else if (n_jobs >= 2 * sms)
    *ctas = std::min(prefill_alone_ctas(tiles, sms), n_jobs - 1);
  return ok();
}

pa_status pa_plan_decode_grid(const int32_t* seq_lens, int32_t n_rows, int32_t num_kv_heads, int32_t sms,
                              int32_t* grid, int32_t* warp_granular) {
  if (!grid || !warp_granular) return fail(PA_ERR_INVALID_ARG, "grid and warp_granular must not be null");
  *grid = 0;
  *warp_granular = 0;
  if (n_rows < 0 || n_rows > pa::kPlanMaxRows || (n_rows > 0 && !seq_lens))
    return fail(PA_ERR_INVALID_ARG, "seq_lens must hold n_rows = %d lengths (at most %d)", n_rows, pa::kPlanMaxRows);
  if (num_kv_heads < 1 || num_kv_heads > 256) return fail(PA_ERR_INVALID_ARG, "num_kv_heads %d outside [1, 256]", num_kv_heads);
  if (sms < 1 || sms > pa::kPlanMaxCtas) return fail(PA_ERR_INVALID_ARG, "sms %d outside [1, %d]", sms, pa::kPlanMaxCtas);
  int32_t max_len = 0;
  for (int32_t r = 0; r < n_rows; ++r) {
    if (seq_lens[r] < 1) return fail(PA_ERR_INVALID_ARG, "row %d: seq_len %d < 1", r, seq_lens[r]);
    max_len = std::max(max_len, seq_lens[r]);
  }
  if (n_rows == 0) return ok();
  std::vector<int32_t> rows((size_t)n_rows), qo_indptr((size_t)n_rows + 1);
  for (int32_t r = 0; r <= n_rows; ++r) {
    if (r < n_rows) rows[(size_t)r] = r;
    qo_indptr[(size_t)r] = r;  // one query per row
  }
  auto plan = std::make_unique<pa::DecodePlan>();
  bool cta_granular = false;
  const int g = choose_decode_plan(rows.data(), n_rows, seq_lens, qo_indptr.data(), 0, num_kv_heads,
                                   grid_cap(n_rows, num_kv_heads, max_len), sms * kDecodeCtasPerSm, false, false,
                                   *plan, cta_granular);
  if (g < 0) return fail(PA_ERR_UNSUPPORTED, "no decode plan within the kernel limits");
  *grid = g;
  *warp_granular = (g > 0 && !cta_granular) ? 1 : 0;
  return ok();
}

pa_status pa_set_decode_fault_injection(int32_t on) {
  if (on != 0 && on != 1) return fail(PA_ERR_INVALID_ARG, "fault injection switch %d (0 or 1)", on);
  g_decode_fault.store(on);
  return ok();
}

int64_t pa_launch_count(void) { return g_launches.load(); }

pa_status pa_trace_enable(int32_t on) {
  std::lock_guard<std::mutex> lk(g_trace_mu);
  g_trace_on = on != 0;
  // create the events up front so that recording costs no event creation
  while (g_trace_on && (int)(g_evpool.size() + 2 * g_trace.size()) < 2 * kTraceCap) {
    cudaEvent_t e = nullptr;
    if (cudaEventCreate(&e) != cudaSuccess) return fail(PA_ERR_CUDA, "creating trace events");
    g_evpool.push_back(e);
  }
  return ok();
}

pa_status pa_trace_read(int32_t* kinds, float* ms, int32_t capacity, int32_t* count) {
  if (!count || capacity < 0 || (capacity > 0 && (!kinds || !ms))) return fail(PA_ERR_INVALID_ARG, "bad arguments");
  std::vector<TraceRec> recs;
  {
    std::lock_guard<std::mutex> lk(g_trace_mu);
    recs.swap(g_trace);
  }
  int32_t n = 0;
  pa_status st = PA_OK;
  for (const TraceRec& r : recs) {
    float t = 0.f;
    cudaError_t e = cudaEventSynchronize(r.end);
    if (e == cudaSuccess) e = cudaEventElapsedTime(&t, r.begin, r.end);
    if (e != cudaSuccess && st == PA_OK) st = fail(PA_ERR_CUDA, "trace event: %s", cudaGetErrorString(e));
    if (n < capacity) {
      kinds[n] = r.kind;
      ms[n] = t;
    }
    ++n;
  }
  {
    std::lock_guard<std::mutex> lk(g_trace_mu);
    for (const TraceRec& r : recs) {
      g_evpool.push_back(r.begin);
      g_evpool.push_back(r.end);
    }
  }
  *count = std::min(n, capacity);
  return st == PA_OK ? ok() : st;
}

}  // extern "C"
