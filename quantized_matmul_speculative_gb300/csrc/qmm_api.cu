// C ABI of libqmm (declared in include/qmm.h): argument validation, the
// variant registry, the dispatcher and the host-side packing helpers.
//
// The dispatcher follows the pages' lesson that the kernel choice must come
// from measurement ("MLX quantized_matmul small-M verify kernels", facts "The
// qmv/qmm switch" and "Maintainers (zcbenz) ... Dispatch-constant tuning was
// tested and refuted"; llama.cpp PR #29869: row thresholds measured per type):
// it looks the shape up in a table generated from a committed benchmark sweep
// (qmm_dispatch_table.inc) and falls back to a rule only for shapes the sweep
// did not cover.
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <vector>

#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "../../include/qmm.h"
#include "qmm_geometry.h"
#include "qmm_internal.h"

namespace qmm {
// Status word of the conversion kernel (this translation unit's; the host
// reads it with the kernels' words in qmm_device_status()): bit 4, a Q4_0 /
// Q8_0 block whose bias -8 d / -128 d is not a finite fp16 (|d| > 8188 /
// 511.75, or d not finite), i.e. a block the affine layout cannot hold.
constexpr unsigned int kStatusGgmlRange = 16u;
static __device__ unsigned int g_qmm_ggml_status = 0;


// Per-(bits, group) launchers, one translation unit each (qmm_mma_inst.cu).
template <int BITS, int GS>
cudaError_t launch_mma_bg(const CallArgs&, const VariantDesc&, int, cudaStream_t);
extern template cudaError_t launch_mma_bg<4, 32>(const CallArgs&, const VariantDesc&, int, cudaStream_t);
extern template cudaError_t launch_mma_bg<4, 64>(const CallArgs&, const VariantDesc&, int, cudaStream_t);
extern template cudaError_t launch_mma_bg<4, 128>(const CallArgs&, const VariantDesc&, int, cudaStream_t);
extern template cudaError_t launch_mma_bg<2, 32>(const CallArgs&, const VariantDesc&, int, cudaStream_t);
extern template cudaError_t launch_mma_bg<2, 64>(const CallArgs&, const VariantDesc&, int, cudaStream_t);
extern template cudaError_t launch_mma_bg<2, 128>(const CallArgs&, const VariantDesc&, int, cudaStream_t);
extern template cudaError_t launch_mma_bg<8, 32>(const CallArgs&, const VariantDesc&, int, cudaStream_t);
extern template cudaError_t launch_mma_bg<8, 64>(const CallArgs&, const VariantDesc&, int, cudaStream_t);
extern template cudaError_t launch_mma_bg<8, 128>(const CallArgs&, const VariantDesc&, int, cudaStream_t);
template <int FMT>
cudaError_t launch_mma_mx(const CallArgs&, const VariantDesc&, int, cudaStream_t);
extern template cudaError_t launch_mma_mx<0>(const CallArgs&, const VariantDesc&, int, cudaStream_t);
extern template cudaError_t launch_mma_mx<1>(const CallArgs&, const VariantDesc&, int, cudaStream_t);
extern template cudaError_t launch_mma_mx<2>(const CallArgs&, const VariantDesc&, int, cudaStream_t);
template <int FMT>
cudaError_t launch_own_mx(const CallArgs&, const VariantDesc&, int, cudaStream_t, bool);
extern template cudaError_t launch_own_mx<0>(const CallArgs&, const VariantDesc&, int, cudaStream_t, bool);
extern template cudaError_t launch_own_mx<1>(const CallArgs&, const VariantDesc&, int, cudaStream_t, bool);
extern template cudaError_t launch_own_mx<2>(const CallArgs&, const VariantDesc&, int, cudaStream_t, bool);

template <int BITS, int GS>
cudaError_t launch_tma_bg(const CallArgs&, const VariantDesc&, int, cudaStream_t);
extern template cudaError_t launch_tma_bg<4, 32>(const CallArgs&, const VariantDesc&, int, cudaStream_t);
extern template cudaError_t launch_tma_bg<4, 64>(const CallArgs&, const VariantDesc&, int, cudaStream_t);
extern template cudaError_t launch_tma_bg<4, 128>(const CallArgs&, const VariantDesc&, int, cudaStream_t);
extern template cudaError_t launch_tma_bg<2, 32>(const CallArgs&, const VariantDesc&, int, cudaStream_t);
extern template cudaError_t launch_tma_bg<2, 64>(const CallArgs&, const VariantDesc&, int, cudaStream_t);
extern template cudaError_t launch_tma_bg<2, 128>(const CallArgs&, const VariantDesc&, int, cudaStream_t);
extern template cudaError_t launch_tma_bg<8, 32>(const CallArgs&, const VariantDesc&, int, cudaStream_t);
extern template cudaError_t launch_tma_bg<8, 64>(const CallArgs&, const VariantDesc&, int, cudaStream_t);
extern template cudaError_t launch_tma_bg<8, 128>(const CallArgs&, const VariantDesc&, int, cudaStream_t);
template <int BITS, int GS>
cudaError_t launch_own_bg(const CallArgs&, const VariantDesc&, int, cudaStream_t, bool);
extern template cudaError_t launch_own_bg<4, 32>(const CallArgs&, const VariantDesc&, int, cudaStream_t, bool);
extern template cudaError_t launch_own_bg<4, 64>(const CallArgs&, const VariantDesc&, int, cudaStream_t, bool);
extern template cudaError_t launch_own_bg<4, 128>(const CallArgs&, const VariantDesc&, int, cudaStream_t, bool);
extern template cudaError_t launch_own_bg<2, 32>(const CallArgs&, const VariantDesc&, int, cudaStream_t, bool);
extern template cudaError_t launch_own_bg<2, 64>(const CallArgs&, const VariantDesc&, int, cudaStream_t, bool);
extern template cudaError_t launch_own_bg<2, 128>(const CallArgs&, const VariantDesc&, int, cudaStream_t, bool);
extern template cudaError_t launch_own_bg<8, 32>(const CallArgs&, const VariantDesc&, int, cudaStream_t, bool);
extern template cudaError_t launch_own_bg<8, 64>(const CallArgs&, const VariantDesc&, int, cudaStream_t, bool);
extern template cudaError_t launch_own_bg<8, 128>(const CallArgs&, const VariantDesc&, int, cudaStream_t, bool);
template <int BITS, int GS>
unsigned int read_device_status(int clear);
extern template unsigned int read_device_status<4, 32>(int);
extern template unsigned int read_device_status<4, 64>(int);
extern template unsigned int read_device_status<4, 128>(int);
extern template unsigned int read_device_status<2, 32>(int);
extern template unsigned int read_device_status<2, 64>(int);
extern template unsigned int read_device_status<2, 128>(int);
extern template unsigned int read_device_status<8, 32>(int);
extern template unsigned int read_device_status<8, 64>(int);
extern template unsigned int read_device_status<8, 128>(int);

namespace {

// mma: {R, WN, WK}; tma: {stages, consumer warps, CTAs per SM}; own: {stages per warp,
// consumer warps, CTAs per SM}.
const VariantDesc kVariants[] = {
    {"mma_r2_wn2_wk4", kFamilyMma, 2, 2, 4},
    {"mma_r1_wn2_wk4", kFamilyMma, 1, 2, 4},
    {"mma_r4_wn1_wk8", kFamilyMma, 4, 1, 8},
    {"tma_w8_2cta", kFamilyTma, 16, 8, 2},
    {"tma_w4_2cta", kFamilyTma, 16, 4, 2},
    {"tma_w8_1cta", kFamilyTma, 16, 8, 1},
    {"tma_w16_1cta", kFamilyTma, 16, 16, 1},
    {"tma_own_w8_d3_1cta", kFamilyOwn, 3, 8, 1},
    {"tma_own_w16_d2_1cta", kFamilyOwn, 2, 16, 1},
    {"tma_own_w8_d3_2cta", kFamilyOwn, 3, 8, 2},
    {"tma_own_w4_d4_2cta", kFamilyOwn, 4, 4, 2},
    {"tma_own_w8_d3_half", kFamilyOwn, 3, 8, 2, 1},
    {"tma_own_w4_d4_half", kFamilyOwn, 4, 4, 2, 1},
    {"tma_own_w8_d2_2cta", kFamilyOwn, 2, 8, 2},
    {"tma_own_w8_d2_1cta", kFamilyOwn, 2, 8, 1},
};
constexpr int kDefaultTma = 3;     // two CTAs per SM
constexpr int kDefaultTma1 = 5;    // one CTA per SM, for wide K-pieces
constexpr int kDefaultOwn = 13;      // tma_own_w8_d2_2cta: the gathered form's default, and the
                                      // fallback where the tma family cannot plan
constexpr int kDefaultOwnWide = 8;   // tma_own_w16_d2_1cta: the same above 12 rows
constexpr int kNumVariants = static_cast<int>(sizeof(kVariants) / sizeof(kVariants[0]));
constexpr int kMaxSplits = 16;

thread_local int g_last_cuda_error = 0;

// One measured choice: the variant and split count for an exact problem shape.
struct TableEntry {
  int M, N, K, bits, gs;
  int variant, splits;
};

const TableEntry kTable[] = {
#include "qmm_dispatch_table.inc"
};
constexpr int kTableSize = static_cast<int>(sizeof(kTable) / sizeof(kTable[0]));

// One measured microscaling choice: the warp-owned variant and split count
// for an exact (format, N, K) at one M (a table of its own: an mxfp4 call and
// an affine 4-bit g32 call of one shape have the same (bits, group)).
struct MxEntry {
  int format, M, N, K;
  int variant, splits;
};

const MxEntry kMxTable[] = {
#include "qmm_mx_table.inc"
};
constexpr int kMxTableSize = static_cast<int>(sizeof(kMxTable) / sizeof(kMxTable[0]));

// The microscaling table's entry: exact M if measured, else the nearest
// measured M of the same (format, N, K) that uses the same number of 8-row
// activation tiles; -1 if the shape was not swept.
int mx_table_lookup(int format, int M, int N, int K, int* splits) {
  int best = -1, best_d = 1 << 30;
  for (int i = 0; i < kMxTableSize; ++i) {
    const MxEntry& e = kMxTable[i];
    if (e.variant < 0 || e.format != format || e.N != N || e.K != K) continue;
    if ((e.M <= 8) != (M <= 8)) continue;
    const int d = e.M > M ? e.M - M : M - e.M;
    if (d < best_d) {
      best_d = d;
      best = i;
    }
  }
  if (best < 0) return -1;
  *splits = kMxTable[best].splits;
  return kMxTable[best].variant;
}

// The dispatch table in use: the compiled-in one, or the file QMM_TABLE names
// (read once per process, in the format of qmm_dispatch_table.inc: one
// "{M, N, K, bits, group, variant, splits}," entry per line, anything after
// "//" ignored).  A QMM_TABLE file that cannot be read or holds no entry is a
// table error: every dispatched call then returns QMM_ERR_TABLE.
struct ActiveTable {
  std::vector<TableEntry> entries;
  bool error = false;
  ActiveTable() {
    const char* path = std::getenv("QMM_TABLE");
    if (path == nullptr || path[0] == '\0') {
      entries.assign(kTable, kTable + kTableSize);
      return;
    }
    FILE* f = std::fopen(path, "r");
    if (f == nullptr) {
      error = true;
      return;
    }
    char line[512];
    while (std::fgets(line, sizeof(line), f) != nullptr) {
      char* c = std::strstr(line, "//");
      if (c != nullptr) *c = '\0';
      TableEntry e;
      if (std::sscanf(line, " { %d , %d , %d , %d , %d , %d , %d }", &e.M, &e.N, &e.K, &e.bits, &e.gs, &e.variant,
                      &e.splits) == 7)
        entries.push_back(e);
    }
    std::fclose(f);
    error = entries.empty();
  }
};

const ActiveTable& active_table() {
  static const ActiveTable t;  // thread-safe one-time initialization
  return t;
}

bool env_flag(const char* name) {
  const char* v = std::getenv(name);
  return v != nullptr && v[0] != '\0' && std::strcmp(v, "0") != 0;
}

// Variant id from QMM_FORCE_VARIANT (a name or an index), or -1.
int forced_variant() {
  const char* v = std::getenv("QMM_FORCE_VARIANT");
  if (v == nullptr || v[0] == '\0') return -1;
  for (int i = 0; i < kNumVariants; ++i)
    if (std::strcmp(v, kVariants[i].name) == 0) return i;
  char* end = nullptr;
  const long id = std::strtol(v, &end, 10);
  if (end != v && *end == '\0' && id >= 0 && id < kNumVariants) return static_cast<int>(id);
  return -2;  // set but unknown
}

int forced_splits() {
  const char* v = std::getenv("QMM_FORCE_SPLITS");
  if (v == nullptr || v[0] == '\0') return -1;
  const int s = std::atoi(v);
  return (s >= 1 && s <= kMaxSplits) ? s : -2;
}

// Split count for shapes the sweep did not cover: enough CTAs for about two per
// SM, at most 8 (portable cluster size), and at least one group per K-warp.
int rule_splits(const VariantDesc& d, int N, int K, int gs) {
  const int rows = variant_rows_per_cta(d);
  const int tiles = (N + rows - 1) / rows;
  const int target = 2 * device_sm_count();
  int s = (target + tiles / 2) / (tiles > 0 ? tiles : 1);
  const int groups = K / gs;
  int cap = groups / d.WK;
  if (cap > 8) cap = 8;
  if (s > cap) s = cap;
  if (s < 1) s = 1;
  return s;
}

// The sweep's entry for this shape: exact M if measured, else the nearest
// measured M of the same (N, K, bits, gs) that uses the same number of 8-row
// activation tiles; -1 if the shape was not swept.
int table_lookup(int M, int N, int K, int bits, int gs, int* splits) {
  const std::vector<TableEntry>& table = active_table().entries;
  int best = -1, best_d = 1 << 30;
  for (int i = 0; i < static_cast<int>(table.size()); ++i) {
    const TableEntry& e = table[i];
    if (e.variant < 0 || e.N != N || e.K != K || e.bits != bits || e.gs != gs) continue;
    if ((e.M <= 8) != (M <= 8)) continue;
    const int d = e.M > M ? e.M - M : M - e.M;
    if (d < best_d) {
      best_d = d;
      best = i;
    }
  }
  if (best < 0) return -1;
  *splits = table[best].splits;
  // host-side fault injection for the error-path tests: the entry reads as corrupt
  const char* inject = std::getenv("QMM_TEST_INJECT");
  if (inject != nullptr && std::strcmp(inject, "bad_table") == 0) return kNumVariants + 1000;
  return table[best].variant;
}

// Cluster size for the TMA family on shapes the sweep did not cover: the
// candidate (8, 4, 2, 1) with the best tile balance over the clusters that fit
// two CTAs per SM, larger clusters first on ties.
int rule_tma_cluster(const CallArgs& a, const VariantDesc& d) {
  // (the gathered form: the tiles of the largest possible union)
  const int tiles = ((a.N + 15) / 16) * (a.rhs != nullptr ? (a.E < a.P ? a.E : a.P) : 1);
  const int sms = device_sm_count();
  int best = -1;
  double best_cost = 1e30;
  for (int c : {8, 4, 2, 1}) {
    if (!tma_supported(a, c, d)) continue;
    int ncl = (d.WK * sms) / c;
    if (ncl > tiles) ncl = tiles;
    if (ncl < 1) ncl = 1;
    // work of the busiest CTA: its tiles times its share of K
    const double per = static_cast<double>((tiles + ncl - 1) / ncl);
    const double cost = per / c + 1e-9 * (8 - c);
    if (cost < best_cost) {
      best_cost = cost;
      best = c;
    }
  }
  return best;
}

// Warp-owned default for shapes the TMA family cannot plan (scale rows that
// are not 16-byte strided): the two-CTA variant up to 12 rows, the one-CTA one
// above (and each as the other's fallback, when shared memory is short), with
// the first cluster size of (4, 2, 1, 8) the planner accepts; -1 if none.
int rule_own(const CallArgs& a, int* splits) {
  const int order[2] = {a.M > 12 ? kDefaultOwnWide : kDefaultOwn, a.M > 12 ? kDefaultOwn : kDefaultOwnWide};
  for (int v : order) {
    for (int c : {4, 2, 1, 8}) {
      if (launch_own(a, kVariants[v], c, nullptr, true) == cudaSuccess) {
        *splits = c;
        return v;
      }
    }
  }
  return -1;
}

// The variant and split count for a call: the table's entry for the shape,
// else the rule-based choice.  -2 for a table error (an unreadable QMM_TABLE
// file, or an entry whose variant or split count is out of range).
int select_variant(const CallArgs& a, int* splits) {
  if (active_table().error) return -2;
  int s = -1;
  const int v = table_lookup(a.M, a.N, a.K, a.bits, a.gs, &s);
  if (v >= 0) {
    if (v >= kNumVariants || s < 1 || s > kMaxSplits) return -2;
    *splits = s;
    return v;
  }
  for (int v : {kDefaultTma, kDefaultTma1}) {
    const int c = rule_tma_cluster(a, kVariants[v]);
    if (c > 0) {
      *splits = c;
      return v;
    }
  }
  const int ov = rule_own(a, splits);
  if (ov >= 0) return ov;
  *splits = rule_splits(kVariants[0], a.N, a.K, a.gs);
  return 0;
}

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

qmm_status fail_cuda(cudaError_t e) {
  g_last_cuda_error = static_cast<int>(e);
  return QMM_ERR_CUDA;
}

}  // namespace

const VariantDesc* variant_desc(int v) { return (v >= 0 && v < kNumVariants) ? &kVariants[v] : nullptr; }
int variant_count() { return kNumVariants; }
int variant_rows_per_cta(const VariantDesc& d) { return d.family == kFamilyMma ? 16 * d.R * d.WN : 16; }

bool tma_supported(const CallArgs& a, int csize, const VariantDesc& d) {
  int gp, pw, bw, nb, mbw;
  if (!tma_geometry(a.K, a.bits, a.gs, csize, &gp, &pw, &bw, &nb, &mbw)) return false;
  if ((reinterpret_cast<uintptr_t>(a.S) | reinterpret_cast<uintptr_t>(a.B)) & 15) return false;
  // the CTA's stages, activations and at least one partial tile must fit
  struct SmemLimits {
    int sm_bytes, optin;
  };
  static const SmemLimits lim = [] {  // one-time, thread-safe initialization
    SmemLimits l{0, 0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&l.sm_bytes, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&l.optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess) {
      cudaGetLastError();
      l = {233472, 232448};  // sm_103a
    }
    return l;
  }();
  const int mp = a.M <= 8 ? 8 : 16;
  // two stages, one tile, every warp a slot; 8-bit codes stage 2g activations per group
  const TmaLayout L(pw, gp, a.bits == 8 ? 2 * a.gs : a.gs, mp, 2, 1, d.WN, mbw);
  return L.total <= tma_smem_budget(lim.sm_bytes, lim.optin, d.WK);
}

cudaError_t launch_own(const CallArgs& a, const VariantDesc& d, int splits, cudaStream_t stream, bool plan_only) {
  switch (a.bits * 1000 + a.gs) {
    case 4032: return launch_own_bg<4, 32>(a, d, splits, stream, plan_only);
    case 4064: return launch_own_bg<4, 64>(a, d, splits, stream, plan_only);
    case 4128: return launch_own_bg<4, 128>(a, d, splits, stream, plan_only);
    case 2032: return launch_own_bg<2, 32>(a, d, splits, stream, plan_only);
    case 2064: return launch_own_bg<2, 64>(a, d, splits, stream, plan_only);
    case 2128: return launch_own_bg<2, 128>(a, d, splits, stream, plan_only);
    case 8032: return launch_own_bg<8, 32>(a, d, splits, stream, plan_only);
    case 8064: return launch_own_bg<8, 64>(a, d, splits, stream, plan_only);
    case 8128: return launch_own_bg<8, 128>(a, d, splits, stream, plan_only);
    default: return cudaErrorNotSupported;
  }
}

cudaError_t launch_tma(const CallArgs& a, const VariantDesc& d, int splits, cudaStream_t stream) {
  switch (a.bits * 1000 + a.gs) {
    case 4032: return launch_tma_bg<4, 32>(a, d, splits, stream);
    case 4064: return launch_tma_bg<4, 64>(a, d, splits, stream);
    case 4128: return launch_tma_bg<4, 128>(a, d, splits, stream);
    case 2032: return launch_tma_bg<2, 32>(a, d, splits, stream);
    case 2064: return launch_tma_bg<2, 64>(a, d, splits, stream);
    case 2128: return launch_tma_bg<2, 128>(a, d, splits, stream);
    case 8032: return launch_tma_bg<8, 32>(a, d, splits, stream);
    case 8064: return launch_tma_bg<8, 64>(a, d, splits, stream);
    case 8128: return launch_tma_bg<8, 128>(a, d, splits, stream);
    default: return cudaErrorInvalidValue;
  }
}

int device_sm_count() {
  static std::mutex mu;
  static int cache[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 148;
  std::lock_guard<std::mutex> lock(mu);
  if (cache[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 148;
    cache[dev] = n;
  }
  return cache[dev];
}

cudaError_t launch_mma(const CallArgs& a, const VariantDesc& d, int splits, cudaStream_t stream) {
  switch (a.bits * 1000 + a.gs) {
    case 4032: return launch_mma_bg<4, 32>(a, d, splits, stream);
    case 4064: return launch_mma_bg<4, 64>(a, d, splits, stream);
    case 4128: return launch_mma_bg<4, 128>(a, d, splits, stream);
    case 2032: return launch_mma_bg<2, 32>(a, d, splits, stream);
    case 2064: return launch_mma_bg<2, 64>(a, d, splits, stream);
    case 2128: return launch_mma_bg<2, 128>(a, d, splits, stream);
    case 8032: return launch_mma_bg<8, 32>(a, d, splits, stream);
    case 8064: return launch_mma_bg<8, 64>(a, d, splits, stream);
    case 8128: return launch_mma_bg<8, 128>(a, d, splits, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace qmm

using namespace qmm;

extern "C" {

const char* qmm_version(void) { return "qmm 0.1 (sm_103a)"; }

const char* qmm_status_string(int s) {
  switch (s) {
    case QMM_OK: return "ok";
    case QMM_ERR_NULL: return "null pointer";
    case QMM_ERR_SHAPE: return "bad shape";
    case QMM_ERR_UNSUPPORTED: return "unsupported bits, group size, variant, split count or output dtype";
    case QMM_ERR_ALIGN: return "misaligned pointer";
    case QMM_ERR_CUDA: return "CUDA runtime error";
    case QMM_ERR_TABLE: return "no usable dispatch table entry";
    default: return "unknown status";
  }
}

int qmm_last_cuda_error(void) { return g_last_cuda_error; }
int qmm_num_variants(void) { return kNumVariants; }
const char* qmm_variant_name(int v) { return (v >= 0 && v < kNumVariants) ? kVariants[v].name : nullptr; }

size_t qmm_packed_words(int64_t N, int64_t K, int bits) {
  if ((bits != 2 && bits != 4 && bits != 8) || N < 0 || K < 0 || (K * bits) % 32 != 0) return 0;
  return static_cast<size_t>(N) * static_cast<size_t>(K * bits / 32);
}

int qmm_select_variant(int M, int N, int K, int bits, int group_size, int* splits) {
  if (M < 1 || M > 16 || N < 1 || K < 1) return -1;
  if ((bits != 2 && bits != 4 && bits != 8) || (group_size != 32 && group_size != 64 && group_size != 128)) return -1;
  if (K % group_size != 0) return -1;
  CallArgs a = {};
  a.M = M;
  a.N = N;
  a.K = K;
  a.bits = bits;
  a.gs = group_size;
  int s = 1;
  const int v = select_variant(a, &s);
  if (v < 0) return -1;
  if (splits) *splits = s;
  return v;
}

unsigned int qmm_device_status(int clear) {
  unsigned int v = 0;
  v |= read_device_status<4, 32>(clear);
  v |= read_device_status<4, 64>(clear);
  v |= read_device_status<4, 128>(clear);
  v |= read_device_status<2, 32>(clear);
  v |= read_device_status<2, 64>(clear);
  v |= read_device_status<2, 128>(clear);
  v |= read_device_status<8, 32>(clear);
  v |= read_device_status<8, 64>(clear);
  v |= read_device_status<8, 128>(clear);
  unsigned int g = 0;
  if (cudaMemcpyFromSymbol(&g, qmm::g_qmm_ggml_status, sizeof(g)) != cudaSuccess) return 0xFFFFFFFFu;
  if (clear && g) {
    const unsigned int zero = 0;
    cudaMemcpyToSymbol(qmm::g_qmm_ggml_status, &zero, sizeof(zero));
  }
  return v | g;
}

}  // extern "C"

namespace {

// One call of either entry point; R is the residual (null: none).
qmm_status run_call(const void* X, const uint32_t* Wq, const void* scales, const void* biases, const void* R, int M,
                    int N, int K, int bits, int group_size, void* Y, int out_dtype, int variant, int splits,
                    void* stream) {
  if (M < 0 || M > 16 || N < 0 || K < 0) return QMM_ERR_SHAPE;
  if (bits != 2 && bits != 4 && bits != 8) return QMM_ERR_UNSUPPORTED;
  if (group_size != 32 && group_size != 64 && group_size != 128) return QMM_ERR_UNSUPPORTED;
  if (out_dtype != QMM_OUT_BF16 && out_dtype != QMM_OUT_F32) return QMM_ERR_UNSUPPORTED;
  if (variant < -1 || variant >= kNumVariants) return QMM_ERR_UNSUPPORTED;
  if (splits == 0 || splits < -1 || splits > kMaxSplits) return QMM_ERR_UNSUPPORTED;
  if (K % group_size != 0) return QMM_ERR_SHAPE;
  if (M == 0 || N == 0) return QMM_OK;
  const size_t esize = out_dtype == QMM_OUT_F32 ? 4 : 2;
  if (Y == nullptr) return QMM_ERR_NULL;
  if (!aligned(Y, esize)) return QMM_ERR_ALIGN;
  const size_t ybytes = static_cast<size_t>(M) * static_cast<size_t>(N) * esize;
  if (R != nullptr) {
    if (!aligned(R, esize)) return QMM_ERR_ALIGN;
    const uintptr_t r0 = reinterpret_cast<uintptr_t>(R), y0 = reinterpret_cast<uintptr_t>(Y);
    if (r0 != y0 && r0 < y0 + ybytes && y0 < r0 + ybytes) return QMM_ERR_SHAPE;  // partial overlap
  }
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (K == 0) {
    // the empty sum: Y = 0, or Y = R
    const cudaError_t e = (R == nullptr) ? cudaMemsetAsync(Y, 0, ybytes, st)
                          : (R == Y)     ? cudaSuccess
                                         : cudaMemcpyAsync(Y, R, ybytes, cudaMemcpyDeviceToDevice, st);
    return e == cudaSuccess ? QMM_OK : fail_cuda(e);
  }
  if (X == nullptr || Wq == nullptr || scales == nullptr || biases == nullptr) return QMM_ERR_NULL;
  if (!aligned(X, 16) || !aligned(Wq, 16) || !aligned(scales, 2) || !aligned(biases, 2)) return QMM_ERR_ALIGN;

  CallArgs a;
  a.X = static_cast<const uint16_t*>(X);
  a.Wq = Wq;
  a.S = static_cast<const uint16_t*>(scales);
  a.B = static_cast<const uint16_t*>(biases);
  a.Y = Y;
  a.R = R;
  a.M = M;
  a.N = N;
  a.K = K;
  a.bits = bits;
  a.gs = group_size;
  a.out_f32 = out_dtype == QMM_OUT_F32;

  int v = variant;
  int s = splits;
  const int fv = forced_variant();
  const int fs = forced_splits();
  if (fv == -2 || fs == -2) return QMM_ERR_UNSUPPORTED;
  if (v < 0 && fv >= 0) v = fv;
  if (s < 0 && fs >= 0) s = fs;
  if (v < 0) {
    int ts = 1;
    v = select_variant(a, &ts);
    if (v < 0) return QMM_ERR_TABLE;
    if (s < 0) s = ts;
    // The table's choice was measured on this shape; if it cannot be planned
    // here (another device, or a resource limit that changed), take the
    // rule-based choice rather than failing.
    const VariantDesc& dt = kVariants[v];
    bool ok = true;
    if (dt.family == kFamilyTma) ok = s >= 1 && tma_supported(a, s, dt);
    if (dt.family == kFamilyOwn) ok = s >= 1 && launch_own(a, dt, s, st, true) == cudaSuccess;
    if (!ok) {
      v = -1;
      for (int dv : {kDefaultTma, kDefaultTma1}) {
        const int c = rule_tma_cluster(a, kVariants[dv]);
        if (c > 0) {
          v = dv;
          s = c;
          break;
        }
      }
      if (v < 0) v = rule_own(a, &s);
      if (v < 0) {
        v = 0;
        s = rule_splits(kVariants[0], a.N, a.K, a.gs);
      }
    }
  }
  const VariantDesc& d = kVariants[v];
  if (s < 0 && d.family == kFamilyOwn) {
    // the first cluster size (4, 2, 1, 8) the planner accepts
    for (int c : {4, 2, 1, 8}) {
      const cudaError_t pe = launch_own(a, d, c, st, true);
      if (pe == cudaSuccess) {
        s = c;
        break;
      }
      if (pe != cudaErrorNotSupported) return fail_cuda(pe);
    }
    if (s < 0) return QMM_ERR_UNSUPPORTED;
  }
  if (s < 0) s = (d.family == kFamilyTma) ? rule_tma_cluster(a, d) : rule_splits(d, N, K, group_size);
  if (d.family == kFamilyTma && (s < 1 || !tma_supported(a, s, d))) return QMM_ERR_UNSUPPORTED;
  if (d.family == kFamilyOwn) {
    if (s < 1) return QMM_ERR_UNSUPPORTED;
    const cudaError_t pe = launch_own(a, d, s, st, true);
    if (pe == cudaErrorNotSupported) return QMM_ERR_UNSUPPORTED;
    if (pe != cudaSuccess) return fail_cuda(pe);
  }
  if (env_flag("QMM_LOG"))
    std::fprintf(stderr, "qmm: M=%d N=%d K=%d bits=%d g=%d -> %s splits=%d\n", M, N, K, bits, group_size, d.name, s);

  // Host-side fault injection for the error-path tests: the launch reports a
  // CUDA error without touching the device.
  const char* inject = std::getenv("QMM_TEST_INJECT");
  if (inject != nullptr && std::strcmp(inject, "launch_fail") == 0) return fail_cuda(cudaErrorLaunchFailure);

  const cudaError_t e = (d.family == kFamilyMma)   ? launch_mma(a, d, s, st)
                        : (d.family == kFamilyTma) ? launch_tma(a, d, s, st)
                        : (d.family == kFamilyOwn) ? launch_own(a, d, s, st, false)
                                                   : cudaErrorInvalidValue;
  return e == cudaSuccess ? QMM_OK : fail_cuda(e);
}

}  // namespace

namespace qmm {

// ggml block -> affine layout (the block layouts are described in qmm.h).
// A CTA of kGgmlThreads threads converts kGgmlBlocks consecutive blocks: it
// first copies their bytes into shared memory with coalesced loads (4-byte
// words, eight in flight per thread, when the span is 4-byte aligned), then
// each thread rewrites blocks t, t + kGgmlThreads.  Codes keep their values
// (Q4) or flip the sign bit (Q8_0: q + 128); the fp16 scale is d; the bias is
// -8 d (Q4_0), m (Q4_1) or -128 d (Q8_0), products by powers of two and so
// exact in fp16.  A block's code words are stored as 16-byte vectors when Wq
// is 16-byte aligned.
constexpr int kGgmlThreads = 256;
constexpr int kGgmlBlocks = 512;

// fp16 bias of a Q4_0 (-8 d) or Q8_0 (-128 d) block: exact (a power-of-two
// multiple) while finite; an infinite or NaN result flags the block.
__device__ __forceinline__ uint16_t ggml_bias(float df, float mult) {
  const uint16_t b = __half_as_ushort(__float2half_rn(mult * df));
  if ((b & 0x7C00u) == 0x7C00u) atomicOr(&g_qmm_ggml_status, kStatusGgmlRange);
  return b;
}

// Four bytes at a 2-byte aligned shared-memory address, as a little-endian word.
__device__ __forceinline__ uint32_t ggml_word(const uint8_t* p) {
  const uint16_t* h = reinterpret_cast<const uint16_t*>(p);
  return static_cast<uint32_t>(h[0]) | (static_cast<uint32_t>(h[1]) << 16);
}

// The low nibbles of the eight bytes of (lo, hi), byte k's at bits 4k.
__device__ __forceinline__ uint32_t ggml_low_nibbles(uint32_t lo, uint32_t hi) {
  auto four = [](uint32_t x) {
    x &= 0x0F0F0F0Fu;
    x = (x | (x >> 4)) & 0x00FF00FFu;
    return (x | (x >> 8)) & 0x0000FFFFu;
  };
  return four(lo) | (four(hi) << 16);
}

// Block i (bytes at blk, 2-byte aligned) into its code words, scale and bias.
// Q4: byte j of the 16 code bytes holds weight j (low nibble) and weight j+16
// (high nibble), so word 0 = the low nibbles of bytes 0..7, word 1 = those of
// bytes 8..15, words 2 and 3 = the high nibbles.
template <int TYPE>
__device__ __forceinline__ void convert_ggml_block(const uint8_t* blk, int64_t i, uint32_t* __restrict__ Wq,
                                                   uint16_t* __restrict__ S, uint16_t* __restrict__ B, bool vec) {
  const uint16_t d = *reinterpret_cast<const uint16_t*>(blk);
  const float df = __half2float(__ushort_as_half(d));
  S[i] = d;
  constexpr int NW = TYPE == 2 ? 8 : 4;
  uint32_t w[NW];
  if constexpr (TYPE == 2) {
#pragma unroll
    for (int k = 0; k < 8; ++k) w[k] = ggml_word(blk + 2 + 4 * k) ^ 0x80808080u;
    B[i] = ggml_bias(df, -128.f);
  } else {
    const uint8_t* qs = blk + (TYPE == 0 ? 2 : 4);
    const uint32_t b0 = ggml_word(qs), b1 = ggml_word(qs + 4), b2 = ggml_word(qs + 8), b3 = ggml_word(qs + 12);
    w[0] = ggml_low_nibbles(b0, b1);
    w[1] = ggml_low_nibbles(b2, b3);
    w[2] = ggml_low_nibbles(b0 >> 4, b1 >> 4);
    w[3] = ggml_low_nibbles(b2 >> 4, b3 >> 4);
    B[i] = (TYPE == 0) ? ggml_bias(df, -8.f) : *reinterpret_cast<const uint16_t*>(blk + 2);
  }
  uint32_t* dst = Wq + i * NW;
  if (vec) {
#pragma unroll
    for (int v = 0; v < NW / 4; ++v) reinterpret_cast<uint4*>(dst)[v] = make_uint4(w[4 * v], w[4 * v + 1], w[4 * v + 2], w[4 * v + 3]);
  } else {
#pragma unroll
    for (int k = 0; k < NW; ++k) dst[k] = w[k];
  }
}

template <int TYPE>
__global__ void __launch_bounds__(kGgmlThreads)
ggml_to_affine_kernel(const uint8_t* __restrict__ blocks, int64_t nblk, uint32_t* __restrict__ Wq,
                      uint16_t* __restrict__ S, uint16_t* __restrict__ B) {
  constexpr int kBytes = TYPE == 0 ? 18 : TYPE == 1 ? 20 : 34;
  __shared__ __align__(16) uint8_t span[kGgmlBlocks * kBytes];
  const int64_t first = static_cast<int64_t>(blockIdx.x) * kGgmlBlocks;
  const int count = static_cast<int>((nblk - first < kGgmlBlocks) ? nblk - first : kGgmlBlocks);
  const uint8_t* src = blocks + first * kBytes;
  const int bytes = count * kBytes;
  int done = 0;
  if ((reinterpret_cast<uintptr_t>(src) & 3) == 0) {
    const int words = bytes >> 2;
    const uint32_t* s32 = reinterpret_cast<const uint32_t*>(src);
    uint32_t* d32 = reinterpret_cast<uint32_t*>(span);
    int w = threadIdx.x;
    for (; w + 7 * kGgmlThreads < words; w += 8 * kGgmlThreads) {  // eight loads in flight
      uint32_t v[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) v[k] = __ldg(s32 + w + k * kGgmlThreads);
#pragma unroll
      for (int k = 0; k < 8; ++k) d32[w + k * kGgmlThreads] = v[k];
    }
    for (; w < words; w += kGgmlThreads) d32[w] = __ldg(s32 + w);
    done = words << 2;
  }
  for (int b = done + threadIdx.x; b < bytes; b += kGgmlThreads) span[b] = __ldg(src + b);
  __syncthreads();
  const bool vec = (reinterpret_cast<uintptr_t>(Wq) & 15) == 0;
  for (int t = threadIdx.x; t < count; t += kGgmlThreads)
    convert_ggml_block<TYPE>(span + t * kBytes, first + t, Wq, S, B, vec);
}

}  // namespace qmm

extern "C" {

qmm_status qmm_from_ggml(int type, const void* blocks, int64_t N, int64_t K, uint32_t* Wq, void* scales, void* biases,
                         void* stream) {
  if (type < QMM_GGML_Q4_0 || type > QMM_GGML_Q8_0) return QMM_ERR_UNSUPPORTED;
  if (N < 0 || K < 0 || K % 32 != 0 || N > (int64_t(1) << 40) / (K + 1)) return QMM_ERR_SHAPE;
  const int64_t nblk = N * (K / 32);
  if (nblk == 0) return QMM_OK;
  if (blocks == nullptr || Wq == nullptr || scales == nullptr || biases == nullptr) return QMM_ERR_NULL;
  if (!aligned(Wq, 4) || !aligned(scales, 2) || !aligned(biases, 2)) return QMM_ERR_ALIGN;
  const int64_t grid = (nblk + qmm::kGgmlBlocks - 1) / qmm::kGgmlBlocks;
  if (grid > 0x7fffffff) return QMM_ERR_SHAPE;
  const uint8_t* blk = static_cast<const uint8_t*>(blocks);
  uint16_t* sp = static_cast<uint16_t*>(scales);
  uint16_t* bp = static_cast<uint16_t*>(biases);
  const cudaStream_t st = static_cast<cudaStream_t>(stream);
  const unsigned int g = static_cast<unsigned int>(grid);
  if (type == QMM_GGML_Q4_0) qmm::ggml_to_affine_kernel<0><<<g, qmm::kGgmlThreads, 0, st>>>(blk, nblk, Wq, sp, bp);
  else if (type == QMM_GGML_Q4_1) qmm::ggml_to_affine_kernel<1><<<g, qmm::kGgmlThreads, 0, st>>>(blk, nblk, Wq, sp, bp);
  else qmm::ggml_to_affine_kernel<2><<<g, qmm::kGgmlThreads, 0, st>>>(blk, nblk, Wq, sp, bp);
  const cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? QMM_OK : fail_cuda(e);
}

qmm_status qmm_small_m_ex(const void* X, const uint32_t* Wq, const void* scales, const void* biases, int M, int N,
                          int K, int bits, int group_size, void* Y, int out_dtype, int variant, int splits,
                          void* stream) {
  return run_call(X, Wq, scales, biases, nullptr, M, N, K, bits, group_size, Y, out_dtype, variant, splits, stream);
}

qmm_status qmm_small_m_residual(const void* X, const uint32_t* Wq, const void* scales, const void* biases,
                                const void* R, int M, int N, int K, int bits, int group_size, void* Y, int out_dtype,
                                int variant, int splits, void* stream) {
  if (M > 0 && N > 0 && R == nullptr) return QMM_ERR_NULL;
  return run_call(X, Wq, scales, biases, R, M, N, K, bits, group_size, Y, out_dtype, variant, splits, stream);
}

qmm_status qmm_gather_small_m(const void* X, const uint32_t* Wq, const void* scales, const void* biases,
                              const int32_t* lhs, const int32_t* rhs, int P, int T, int E, int N, int K, int bits,
                              int group_size, void* Y, int out_dtype, int variant, int splits, void* stream) {
  if (P < 0 || P > kMaxGatherEntries || T < 0 || E < 0 || N < 0 || K < 0) return QMM_ERR_SHAPE;
  if (bits != 2 && bits != 4 && bits != 8) return QMM_ERR_UNSUPPORTED;
  if (group_size != 32 && group_size != 64 && group_size != 128) return QMM_ERR_UNSUPPORTED;
  if (out_dtype != QMM_OUT_BF16 && out_dtype != QMM_OUT_F32) return QMM_ERR_UNSUPPORTED;
  if (variant < -1 || variant >= kNumVariants) return QMM_ERR_UNSUPPORTED;
  if (splits == 0 || splits < -1 || splits > kMaxSplits) return QMM_ERR_UNSUPPORTED;
  if (K % group_size != 0) return QMM_ERR_SHAPE;
  if (P == 0 || N == 0) return QMM_OK;
  const size_t esize = out_dtype == QMM_OUT_F32 ? 4 : 2;
  if (Y == nullptr) return QMM_ERR_NULL;
  if (!aligned(Y, esize)) return QMM_ERR_ALIGN;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (K == 0) {
    const cudaError_t e = cudaMemsetAsync(Y, 0, static_cast<size_t>(P) * static_cast<size_t>(N) * esize, st);
    return e == cudaSuccess ? QMM_OK : fail_cuda(e);
  }
  if (T < 1 || E < 1) return QMM_ERR_SHAPE;
  if (X == nullptr || Wq == nullptr || scales == nullptr || biases == nullptr || lhs == nullptr || rhs == nullptr)
    return QMM_ERR_NULL;
  if (!aligned(X, 16) || !aligned(Wq, 16) || !aligned(scales, 2) || !aligned(biases, 2) || !aligned(lhs, 4) ||
      !aligned(rhs, 4))
    return QMM_ERR_ALIGN;

  CallArgs a;
  a.X = static_cast<const uint16_t*>(X);
  a.Wq = Wq;
  a.S = static_cast<const uint16_t*>(scales);
  a.B = static_cast<const uint16_t*>(biases);
  a.Y = Y;
  a.R = nullptr;
  a.M = 0;
  a.N = N;
  a.K = K;
  a.bits = bits;
  a.gs = group_size;
  a.out_f32 = out_dtype == QMM_OUT_F32;
  a.lhs = lhs;
  a.rhs = rhs;
  a.P = P;
  a.T = T;
  a.E = E;
  const int fv = forced_variant();
  if (variant < 0 && fv >= 0) variant = fv;

  // The warp-owned family (the default when it can plan the shape, measured
  // about twice as fast as the mma family on the 128-expert top-8 stack):
  // every token row against each expert of the union, like the tma variants,
  // with per-warp copy rings and no reduction rounds.  Cluster sizes from 1
  // up: a union of a few experts has few tiles, and splitting K over a
  // cluster then only adds reduction (on the 128-expert top-8 gate+up stack,
  // T = 1, 2, 4, 8: 11.7 / 14.8 / 18.5 / 31.1 us unsplit against 12.1 / 15.4 /
  // 20.6 / 34.1 with clusters of 4).
  const bool own_forced = variant >= 0 && kVariants[variant].family == kFamilyOwn;
  if (variant < 0 && T <= 16) {
    CallArgs ao = a;
    ao.M = T;
    const VariantDesc& dd = kVariants[kDefaultOwn];
    for (int cc : {1, 2, 4, 8}) {
      if (splits > 0 && cc != splits) continue;
      const cudaError_t pe = launch_own(ao, dd, cc, st, true);
      if (pe == cudaErrorNotSupported) continue;
      if (pe != cudaSuccess) return fail_cuda(pe);
      if (env_flag("QMM_LOG"))
        std::fprintf(stderr, "qmm gather: P=%d T=%d E=%d N=%d K=%d bits=%d g=%d -> %s splits=%d\n", P, T, E, N, K,
                     bits, group_size, dd.name, cc);
      const cudaError_t e = launch_own(ao, dd, cc, st, false);
      return e == cudaSuccess ? QMM_OK : fail_cuda(e);
    }
  }
  if (own_forced) {
    if (T > 16) return QMM_ERR_UNSUPPORTED;
    CallArgs ao = a;
    ao.M = T;
    const VariantDesc& dd = kVariants[variant];
    int c = splits;
    if (c < 0) {
      for (int cc : {4, 2, 1, 8}) {
        const cudaError_t pe = launch_own(ao, dd, cc, st, true);
        if (pe == cudaSuccess) {
          c = cc;
          break;
        }
        if (pe != cudaErrorNotSupported) return fail_cuda(pe);
      }
      if (c < 0) return QMM_ERR_UNSUPPORTED;
    }
    if (env_flag("QMM_LOG"))
      std::fprintf(stderr, "qmm gather: P=%d T=%d E=%d N=%d K=%d bits=%d g=%d -> %s splits=%d\n", P, T, E, N, K,
                   bits, group_size, dd.name, c);
    const cudaError_t e = launch_own(ao, dd, c, st, false);
    if (e == cudaSuccess) return QMM_OK;
    if (e == cudaErrorNotSupported) return QMM_ERR_UNSUPPORTED;
    return fail_cuda(e);
  }

  // A tma variant (forced) computes every token row against each expert of
  // the union (T <= 16 rows staged once) under the TMA shape rules (slower on
  // large unions: many reduction rounds); the mma family (the fallback) takes
  // each expert's own entries (at most 8 or 16 of them).
  const bool tma_forced = variant >= 0 && kVariants[variant].family == kFamilyTma;
  if (T <= 16 && tma_forced) {
    CallArgs at = a;
    at.M = T;
    const VariantDesc& dd = kVariants[variant];
    if (P > 32 * (dd.WN + 1)) return QMM_ERR_UNSUPPORTED;
    const int c = splits > 0 ? (tma_supported(at, splits, dd) ? splits : -1) : rule_tma_cluster(at, dd);
    if (c < 1) return QMM_ERR_UNSUPPORTED;
    if (env_flag("QMM_LOG"))
      std::fprintf(stderr, "qmm gather: P=%d T=%d E=%d N=%d K=%d bits=%d g=%d -> %s splits=%d\n", P, T, E, N, K,
                   bits, group_size, dd.name, c);
    const cudaError_t e = launch_tma(at, dd, c, st);
    if (e == cudaSuccess) return QMM_OK;
    if (e == cudaErrorInvalidValue) return QMM_ERR_UNSUPPORTED;
    return fail_cuda(e);
  } else if (tma_forced) {
    return QMM_ERR_UNSUPPORTED;
  }
  a.M = (T <= 8 || P <= 8) ? 8 : 16;  // entries one expert may take: the activation tile
  const VariantDesc& d = kVariants[variant < 0 ? 0 : variant];
  int s = splits;
  if (s < 0) {
    // about two CTAs per SM over the tiles of every possible expert of the union
    const int slots = E < P ? E : P;
    const int rows = variant_rows_per_cta(d);
    const int64_t ctas = static_cast<int64_t>((N + rows - 1) / rows) * slots;
    const int64_t target = 2 * static_cast<int64_t>(device_sm_count());
    s = static_cast<int>((target + ctas - 1) / ctas);
    int cap = (K / group_size) / d.WK;
    if (cap > 8) cap = 8;
    if (s > cap) s = cap;
    if (s < 1) s = 1;
  }
  if (env_flag("QMM_LOG"))
    std::fprintf(stderr, "qmm gather: P=%d T=%d E=%d N=%d K=%d bits=%d g=%d -> %s splits=%d\n", P, T, E, N, K, bits,
                 group_size, d.name, s);
  const cudaError_t e = launch_mma(a, d, s, st);
  return e == cudaSuccess ? QMM_OK : fail_cuda(e);
}

qmm_status qmm_small_m_mx(const void* X, const uint32_t* Wq, const uint8_t* scales, int M, int N, int K, int format,
                          void* Y, int out_dtype, int variant, int splits, void* stream) {
  if (M < 0 || M > 16 || N < 0 || K < 0) return QMM_ERR_SHAPE;
  if (format != QMM_MXFP4 && format != QMM_MXFP8 && format != QMM_NVFP4) return QMM_ERR_UNSUPPORTED;
  if (out_dtype != QMM_OUT_BF16 && out_dtype != QMM_OUT_F32) return QMM_ERR_UNSUPPORTED;
  if (variant < -1 || variant >= kNumVariants || (variant >= 0 && kVariants[variant].family == kFamilyTma))
    return QMM_ERR_UNSUPPORTED;
  if (splits == 0 || splits < -1 || splits > kMaxSplits) return QMM_ERR_UNSUPPORTED;
  if (K % 32 != 0) return QMM_ERR_SHAPE;
  if (M == 0 || N == 0) return QMM_OK;
  const size_t esize = out_dtype == QMM_OUT_F32 ? 4 : 2;
  if (Y == nullptr) return QMM_ERR_NULL;
  if (!aligned(Y, esize)) return QMM_ERR_ALIGN;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (K == 0) {
    const cudaError_t e = cudaMemsetAsync(Y, 0, static_cast<size_t>(M) * static_cast<size_t>(N) * esize, st);
    return e == cudaSuccess ? QMM_OK : fail_cuda(e);
  }
  if (X == nullptr || Wq == nullptr || scales == nullptr) return QMM_ERR_NULL;
  if (!aligned(X, 16) || !aligned(Wq, 16)) return QMM_ERR_ALIGN;
  CallArgs a;
  a.X = static_cast<const uint16_t*>(X);
  a.Wq = Wq;
  a.S = nullptr;
  a.B = nullptr;
  a.S8 = scales;
  a.Y = Y;
  a.R = nullptr;
  a.M = M;
  a.N = N;
  a.K = K;
  a.bits = format == QMM_MXFP8 ? 8 : 4;
  a.gs = format == QMM_NVFP4 ? 16 : 32;
  a.out_f32 = out_dtype == QMM_OUT_F32;
  // The warp-owned family when it can plan the shape, else mma.  Variant -1:
  // the microscaling table's choice for a swept (format, N, K) (nearest M of
  // the same activation-tile class), else tma_own_w8_d2_2cta, or
  // tma_own_w16_d2_1cta above 12 rows, with the first cluster size of
  // (4, 2, 1, 8) that plans; or a forced warp-owned variant.
  auto own_mx = [&](const VariantDesc& dd, int cc, bool plan_only) {
    return (format == QMM_MXFP4)   ? launch_own_mx<0>(a, dd, cc, st, plan_only)
           : (format == QMM_MXFP8) ? launch_own_mx<1>(a, dd, cc, st, plan_only)
                                   : launch_own_mx<2>(a, dd, cc, st, plan_only);
  };
  if (variant < 0 && splits <= 0) {
    int ts = 0;
    const int tv = mx_table_lookup(format, M, N, K, &ts);
    if (tv >= 0 && tv < kNumVariants && kVariants[tv].family == kFamilyOwn &&
        own_mx(kVariants[tv], ts, true) == cudaSuccess) {
      if (env_flag("QMM_LOG"))
        std::fprintf(stderr, "qmm mx: M=%d N=%d K=%d format=%d -> %s splits=%d (table)\n", M, N, K, format,
                     kVariants[tv].name, ts);
      const cudaError_t e = own_mx(kVariants[tv], ts, false);
      return e == cudaSuccess ? QMM_OK : fail_cuda(e);
    }
  }
  const bool own_forced = variant >= 0 && kVariants[variant].family == kFamilyOwn;
  if (variant < 0 || own_forced) {
    const VariantDesc& dd = kVariants[own_forced ? variant : (M > 12 ? kDefaultOwnWide : kDefaultOwn)];
    for (int cc : {4, 2, 1, 8}) {
      if (splits > 0 && cc != splits) continue;
      const cudaError_t pe = own_mx(dd, cc, true);
      if (pe == cudaErrorNotSupported) continue;
      if (pe != cudaSuccess) return fail_cuda(pe);
      if (env_flag("QMM_LOG"))
        std::fprintf(stderr, "qmm mx: M=%d N=%d K=%d format=%d -> %s splits=%d\n", M, N, K, format, dd.name, cc);
      const cudaError_t e = own_mx(dd, cc, false);
      return e == cudaSuccess ? QMM_OK : fail_cuda(e);
    }
    if (own_forced) return QMM_ERR_UNSUPPORTED;
  }
  const VariantDesc& d = kVariants[variant < 0 ? 0 : variant];
  const int s = splits > 0 ? splits : rule_splits(d, N, K, a.gs);
  if (env_flag("QMM_LOG"))
    std::fprintf(stderr, "qmm mx: M=%d N=%d K=%d format=%d -> %s splits=%d\n", M, N, K, format, d.name, s);
  const cudaError_t e = (format == QMM_MXFP4)   ? launch_mma_mx<0>(a, d, s, st)
                        : (format == QMM_MXFP8) ? launch_mma_mx<1>(a, d, s, st)
                                                : launch_mma_mx<2>(a, d, s, st);
  return e == cudaSuccess ? QMM_OK : fail_cuda(e);
}

qmm_status qmm_small_m(const void* X, const uint32_t* Wq, const void* scales, const void* biases, int M, int N, int K,
                       int bits, int group_size, void* Y, void* stream) {
  return qmm_small_m_ex(X, Wq, scales, biases, M, N, K, bits, group_size, Y, QMM_OUT_BF16, -1, -1, stream);
}

// Packing, host side.  Word j of a row collects codes j*per .. j*per+per-1,
// code i of the word at bits [bits*i, bits*i + bits).
qmm_status qmm_pack(const uint8_t* q, int64_t N, int64_t K, int bits, uint32_t* Wq) {
  if ((N > 0 && K > 0) && (q == nullptr || Wq == nullptr)) return QMM_ERR_NULL;
  if (bits != 2 && bits != 4 && bits != 8) return QMM_ERR_UNSUPPORTED;
  if (N < 0 || K < 0 || (K * bits) % 32 != 0) return QMM_ERR_SHAPE;
  const int per = 32 / bits;
  const uint32_t limit = 1u << bits;
  const uint8_t* src = q;
  uint32_t* dst = Wq;
  const int64_t words = N * (K / per);
  for (int64_t w = 0; w < words; ++w) {
    uint32_t acc = 0;
    for (int i = per - 1; i >= 0; --i) {
      const uint32_t c = src[i];
      if (c >= limit) return QMM_ERR_SHAPE;
      acc = (acc << bits) | c;
    }
    *dst++ = acc;
    src += per;
  }
  return QMM_OK;
}

qmm_status qmm_unpack(const uint32_t* Wq, int64_t N, int64_t K, int bits, uint8_t* q) {
  if ((N > 0 && K > 0) && (q == nullptr || Wq == nullptr)) return QMM_ERR_NULL;
  if (bits != 2 && bits != 4 && bits != 8) return QMM_ERR_UNSUPPORTED;
  if (N < 0 || K < 0 || (K * bits) % 32 != 0) return QMM_ERR_SHAPE;
  const int per = 32 / bits;
  const uint32_t mask = (1u << bits) - 1u;
  const int64_t words = N * (K / per);
  for (int64_t w = 0; w < words; ++w) {
    uint32_t word = Wq[w];
    for (int i = 0; i < per; ++i) {
      *q++ = static_cast<uint8_t>(word & mask);
      word >>= bits;
    }
  }
  return QMM_OK;
}

// The kernels read the canonical layout itself (the k-permutation the MMA
// fragments need is applied to the activations in shared memory), so the
// native layout is the canonical one and converting is a copy.
static qmm_status layout_copy(const uint32_t* src, int64_t N, int64_t K, int bits, uint32_t* dst, void* stream) {
  if (bits != 2 && bits != 4 && bits != 8) return QMM_ERR_UNSUPPORTED;
  if (N < 0 || K < 0 || (K * bits) % 32 != 0) return QMM_ERR_SHAPE;
  const size_t bytes = static_cast<size_t>(N) * static_cast<size_t>(K) * static_cast<size_t>(bits) / 8;
  if (bytes == 0) return QMM_OK;
  if (src == nullptr || dst == nullptr) return QMM_ERR_NULL;
  if (src == dst) return QMM_OK;
  const cudaError_t e =
      cudaMemcpyAsync(dst, src, bytes, cudaMemcpyDeviceToDevice, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? QMM_OK : fail_cuda(e);
}

qmm_status qmm_repack(const uint32_t* Wq, int64_t N, int64_t K, int bits, uint32_t* Wq_native, void* stream) {
  return layout_copy(Wq, N, K, bits, Wq_native, stream);
}

qmm_status qmm_unrepack(const uint32_t* Wq_native, int64_t N, int64_t K, int bits, uint32_t* Wq, void* stream) {
  return layout_copy(Wq_native, N, K, bits, Wq, stream);
}

}  // extern "C"
