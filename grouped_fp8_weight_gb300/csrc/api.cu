// C-ABI entry points: argument validation, the expert schedule, TMA tensor
// maps and kernel launches.  Allocation: one status word per device on first
// use and, per FP8 call, stream-ordered scratch for the packed scale factors
// from a memory pool this library owns (returned to the pool on the same
// stream once the GEMM is queued; the pool keeps it for the next call).
#include <algorithm>
#include <cstddef>
#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <memory>
#include <mutex>
#include <string>
#include <vector>

#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include "dg_wgrad.h"
#include "grouped_plan.h"
#include "wgrad_params.h"

static_assert(DG_MAX_GROUPS == dg::kMaxGroups, "group limit mismatch");

#ifdef DG_KERNEL_TIMERS
// Profiling builds only: device buffer receiving the kernel's per-role cycle
// counters (32 per CTA).
static unsigned long long *g_timers = nullptr;
extern "C" void dg_debug_set_timers(unsigned long long *p) { g_timers = p; }
#endif

namespace {

thread_local std::string g_err;

dg_status fail(dg_status s, const char *fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_err = buf;
  return s;
}

dg_status ok() {
  g_err.clear();
  return DG_OK;
}

struct DeviceState {
  bool init = false;
  bool arch_ok = false;
  int major = 0, minor = 0;
  int sms = 0;
  dg::DevStatus *status = nullptr;
  cudaMemPool_t pool = nullptr;   // packed scale-factor scratch
};

constexpr int kMaxDevices = 64;
std::mutex g_mu;
DeviceState g_dev[kMaxDevices];

dg_status device_state(DeviceState **out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return fail(DG_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
  if (dev < 0 || dev >= kMaxDevices) return fail(DG_ERR_UNSUPPORTED, "device index %d", dev);
  if (dg::tensor_map_encoder() == nullptr)
    return fail(DG_ERR_CUDA, "cuTensorMapEncodeTiled not available");
  std::lock_guard<std::mutex> lock(g_mu);
  DeviceState &st = g_dev[dev];
  if (!st.init) {
    if ((e = cudaDeviceGetAttribute(&st.major, cudaDevAttrComputeCapabilityMajor, dev)) !=
            cudaSuccess ||
        (e = cudaDeviceGetAttribute(&st.minor, cudaDevAttrComputeCapabilityMinor, dev)) !=
            cudaSuccess ||
        (e = cudaDeviceGetAttribute(&st.sms, cudaDevAttrMultiProcessorCount, dev)) !=
            cudaSuccess)
      return fail(DG_ERR_CUDA, "device query: %s", cudaGetErrorString(e));
    st.arch_ok = (st.major == 10 && st.minor == 3);
    if (st.arch_ok) {
      if ((e = cudaMalloc(&st.status, sizeof(dg::DevStatus))) != cudaSuccess ||
          (e = cudaMemset(st.status, 0, sizeof(dg::DevStatus))) != cudaSuccess)
        return fail(DG_ERR_CUDA, "status word: %s", cudaGetErrorString(e));
      cudaMemPoolProps props{};
      props.allocType = cudaMemAllocationTypePinned;
      props.handleTypes = cudaMemHandleTypeNone;
      props.location.type = cudaMemLocationTypeDevice;
      props.location.id = dev;
      uint64_t keep = ~0ull;   // keep freed blocks for reuse instead of releasing them
      if ((e = cudaMemPoolCreate(&st.pool, &props)) != cudaSuccess ||
          (e = cudaMemPoolSetAttribute(st.pool, cudaMemPoolAttrReleaseThreshold, &keep)) !=
              cudaSuccess)
        return fail(DG_ERR_CUDA, "memory pool: %s", cudaGetErrorString(e));
    }
    st.init = true;
  }
  if (!st.arch_ok)
    return fail(DG_ERR_UNSUPPORTED, "device is sm_%d%d; this library is built for sm_103a only",
                st.major, st.minor);
  *out = &st;
  return DG_OK;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// DG_LOG=1 in the environment (read at each call): each GEMM call prints its
// plan to stderr.
bool log_enabled() {
  const char *v = std::getenv("DG_LOG");
  return v != nullptr && *v != '\0' && *v != '0';
}

dg_status encode(CUtensorMap *m, CUtensorMapDataType dt, const void *ptr, int rank,
                 const uint64_t *dims, const uint64_t *strides_bytes, const uint32_t *box,
                 CUtensorMapSwizzle sw, CUtensorMapL2promotion l2, const char *what) {
  cuuint64_t gd[3];
  cuuint64_t gs[2];
  cuuint32_t bx[3], es[3];
  for (int i = 0; i < rank; ++i) {
    gd[i] = dims[i];
    bx[i] = box[i];
    es[i] = 1;
  }
  for (int i = 0; i + 1 < rank; ++i) gs[i] = strides_bytes[i];
  PFN_cuTensorMapEncodeTiled_v12000 enc = dg::tensor_map_encoder();
  if (enc == nullptr) return fail(DG_ERR_CUDA, "cuTensorMapEncodeTiled not available");
  CUresult r = enc(m, dt, static_cast<cuuint32_t>(rank), const_cast<void *>(ptr), gd, gs, bx, es,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, sw, l2, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(DG_ERR_CUDA, "tensor map for %s failed (%d)", what, (int)r);
  return DG_OK;
}

}  // namespace

namespace dg {

cudaError_t noalloc_take_status(DevStatus *out, bool *present);   // noalloc.cu

dg_status failf(dg_status s, const char *fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_err = buf;
  return s;
}

// Lets the allocation-free entry point (noalloc.cu) report through dg_last_error.
void set_last_error(const char *msg) { g_err = (msg != nullptr) ? msg : ""; }

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static const PFN_cuTensorMapEncodeTiled_v12000 enc = [] {
    void *fn = nullptr;
    cudaDriverEntryPointQueryResult q{};
    const cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                                           cudaEnableDefault, &q);
    return (e == cudaSuccess && q == cudaDriverEntryPointSuccess)
               ? reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn)
               : nullptr;
  }();
  return enc;
}

uint64_t wait_limit_ns() {
  // DG_WAIT_LIMIT_US (microseconds) takes precedence over DG_WAIT_LIMIT_MS.
  const char *us = std::getenv("DG_WAIT_LIMIT_US");
  if (us != nullptr && *us) {
    char *end = nullptr;
    const long long v = std::strtoll(us, &end, 10);
    if (end != us && v > 0) return static_cast<uint64_t>(v) * 1000ull;
  }
  const char *s = std::getenv("DG_WAIT_LIMIT_MS");
  long long ms = 4000;
  if (s != nullptr && *s) {
    char *end = nullptr;
    const long long v = std::strtoll(s, &end, 10);
    if (end != s && v > 0) ms = v;
  }
  return static_cast<uint64_t>(ms) * 1000000ull;
}

bool deterministic_requested() {
  const char *v = std::getenv("DG_DETERMINISTIC");
  return v != nullptr && *v != '\0' && *v != '0';
}

bool pdl_requested() {
  const char *v = std::getenv("DG_PDL");
  return v == nullptr || *v != '0';
}

// DG_MIXED_TILES in the environment (read at each call): 0 keeps every FP8
// tile 224 columns wide; a positive number is the percentage of the narrow
// tiles' count that the wide tiles' lane-0 turns may reach (see
// grouped_schedule).  -1 when unset: the default for the output mode.
static int mixed_tiles_percent() {
  const char *v = std::getenv("DG_MIXED_TILES");
  if (v == nullptr || *v == '\0') return -1;
  const int pct = std::atoi(v);
  return pct < 0 ? 0 : pct;
}

dg_status grouped_validate(const GroupedArgs &x) {
  const char *fn = x.fn;
  if (x.G < 0) return fail(DG_ERR_INVALID_ARG, "%s: G = %d < 0", fn, x.G);
  if (x.G > DG_MAX_GROUPS)
    return fail(DG_ERR_UNSUPPORTED, "%s: G = %d above the maximum of %d experts", fn, x.G,
                DG_MAX_GROUPS);
  const int mult = x.fp8 ? 16 : 8;
  if (x.M <= 0 || x.N <= 0 || x.M % mult || x.N % mult)
    return fail(DG_ERR_INVALID_ARG, "%s: M = %d, N = %d must be positive multiples of %d", fn,
                x.M, x.N, mult);
  if (x.sum_k < 0) return fail(DG_ERR_INVALID_ARG, "%s: sum_k < 0", fn);
  if (x.sum_k > (int64_t)0x7FFFFF00)
    return fail(DG_ERR_UNSUPPORTED, "%s: sum_k above the maximum of 2^31 - 256", fn);
  if (x.fp8 && x.gran_k != 32 && x.gran_k != 128)
    return fail(DG_ERR_INVALID_ARG, "%s: gran_k = %d (must be 32 or 128)", fn, x.gran_k);
  if (x.d_dtype != DG_F32 && x.d_dtype != DG_BF16)
    return fail(DG_ERR_INVALID_ARG, "%s: unknown output dtype %d", fn, (int)x.d_dtype);
  if (x.d_dtype == DG_BF16 && x.c != nullptr)
    return fail(DG_ERR_INVALID_ARG, "%s: an accumulator needs FP32 output", fn);
  if (x.G == 0) {
    if (x.sum_k != 0)
      return fail(DG_ERR_INVALID_ARG, "%s: G = 0 but sum_k = %lld", fn, (long long)x.sum_k);
    return DG_OK;
  }
  if (x.ks_host == nullptr || x.ks_dev == nullptr)
    return fail(DG_ERR_INVALID_ARG, "%s: ks_host and ks_dev are required", fn);
  int64_t total = 0;
  for (int e = 0; e < x.G; ++e) {
    const int k = x.ks_host[e];
    if (k < 0) return fail(DG_ERR_INVALID_ARG, "%s: ks[%d] = %d < 0", fn, e, k);
    if (x.fp8 && k % 128)
      return fail(DG_ERR_INVALID_ARG, "%s: ks[%d] = %d is not a multiple of 128", fn, e, k);
    total += k;
  }
  if (total != x.sum_k)
    return fail(DG_ERR_INVALID_ARG, "%s: sum of ks (%lld) != sum_k (%lld)", fn,
                (long long)total, (long long)x.sum_k);
  if (x.d == nullptr || !aligned16(x.d))
    return fail(DG_ERR_INVALID_ARG, "%s: d must be a 16-byte aligned device pointer", fn);
  if (x.c != nullptr && x.c != x.d && !aligned16(x.c))
    return fail(DG_ERR_INVALID_ARG, "%s: c must be 16-byte aligned", fn);
  if (x.sum_k > 0) {
    if (x.a == nullptr || x.b == nullptr || !aligned16(x.a) || !aligned16(x.b))
      return fail(DG_ERR_INVALID_ARG, "%s: a and b must be 16-byte aligned device pointers", fn);
    if (x.fp8 && (x.sfa == nullptr || x.sfb == nullptr || !aligned16(x.sfa) ||
                  !aligned16(x.sfb)))
      return fail(DG_ERR_INVALID_ARG, "%s: sfa and sfb must be 16-byte aligned device pointers",
                  fn);
  }
  return DG_OK;
}

void grouped_schedule(const GroupedArgs &x, int sms, WgradParams &p, PackParams &pk,
                      GroupedPlan &g) {
  // Clear everything but the per-entry tables; the entries in use are written
  // below and the kernels and the pack pass read no others.
  std::memset(&p, 0, offsetof(WgradParams, sched));
  std::memset(&pk, 0, offsetof(PackParams, g_off));
  // FP8 with N not a multiple of 224 but M one (the down-projection's 7168 x
  // 2048): compute D^T tiles instead, so that the 224-wide tile runs along M
  // with no ragged edge and the 256-row side along N.
  g.trans = x.fp8 && (x.N % 224 != 0) && (x.M % 224 == 0);
  const int Mk = g.trans ? x.N : x.M, Nk = g.trans ? x.M : x.N;   // the kernel's M and N
  g.ksfa = g.trans ? x.sfb : x.sfa;
  g.ksfb = g.trans ? x.sfa : x.sfb;
  g.bn = x.fp8 ? fp8_pick_block_n(Nk) : bf16_pick_block_n(Nk);
  const int bn = g.bn;
  const int tpg = ((Mk + kPairM - 1) / kPairM) * ((Nk + bn - 1) / bn);
  const bool reduce = (x.c == x.d) && x.d_dtype == DG_F32;   // D += acc in place

  // Entries: (expert, first token, tokens); fixed-size per-thread storage, so
  // that planning takes no heap memory.
  struct Entry {
    int expert;
    int64_t k_off;
    int k_len;
  };
  static thread_local Entry ents[2 * kMaxGroups];
  static thread_local Entry split[kMaxGroups];
  static thread_local int64_t off[kMaxGroups + 1];
  int n = 0;
  off[0] = 0;
  for (int e = 0; e < x.G; ++e) off[e + 1] = off[e] + x.ks_host[e];
  for (int e = 0; e < x.G; ++e)
    if (x.ks_host[e] > 0) ents[n++] = Entry{e, off[e], x.ks_host[e]};
  // In-place accumulation: experts much longer than a CTA pair's fair share of
  // the work are split along K into several entries, each adding its part
  // into D (exact by linearity; the order of the FP32 additions then depends
  // on timing).  A pair's fair share is (stages x tiles) / pairs; entries are
  // capped at a quarter of it, in whole scale groups for FP8.
  if (reduce && n > 0 && sms > 0 && !deterministic_requested()) {
    const int bk = x.fp8 ? 128 : 64;            // tokens per stage
    const int unit = x.fp8 ? 4 : 1;             // stages per split unit
    int64_t total = 0;
    for (int i = 0; i < n; ++i) total += (ents[i].k_len + bk - 1) / bk;
    const int64_t share = total * tpg / std::max(1, sms / 2);
    const int64_t cap = std::max<int64_t>(8, share / 4);   // stages per entry
    int ns = 0;
    bool fits = true;
    for (int i = 0; i < n && fits; ++i) {
      const Entry &en = ents[i];
      const int64_t st = (en.k_len + bk - 1) / bk;
      if (st <= cap) {
        if (ns == kMaxGroups) { fits = false; break; }
        split[ns++] = en;
        continue;
      }
      const int64_t parts = (st + cap - 1) / cap;
      int64_t per = (st + parts - 1) / parts;
      per = (per + unit - 1) / unit * unit;
      for (int64_t s0 = 0; s0 < st; s0 += per) {
        if (ns == kMaxGroups) { fits = false; break; }
        const int64_t t0 = s0 * bk;
        const int64_t t1 = std::min<int64_t>(en.k_len, (s0 + per) * bk);
        split[ns++] = Entry{en.expert, en.k_off + t0, static_cast<int>(t1 - t0)};
      }
    }
    if (fits) {
      for (int i = 0; i < ns; ++i) ents[i] = split[i];
      n = ns;
    }
  }
  std::stable_sort(ents, ents + n, [](const Entry &u, const Entry &v) { return u.k_len > v.k_len; });
  g.n_mma = n;
  if (x.c != x.d)   // no accumulator, or a separate one: empty experts still write D
    for (int e = 0; e < x.G; ++e)
      if (x.ks_host[e] == 0) ents[n++] = Entry{e, off[e], 0};
  g.n_sched = n;
  for (int i = 0; i < n; ++i) {
    p.sched[i].expert = ents[i].expert;
    p.sched[i].k_off = static_cast<int>(ents[i].k_off);
    p.sched[i].k_len = ents[i].k_len;
    p.sched[i].k_exp = x.ks_host[ents[i].expert];
  }
  p.M = Mk;
  p.N = Nk;
  p.G = x.G;
  p.m_tiles = (Mk + kPairM - 1) / kPairM;
  p.n_tiles = (Nk + bn - 1) / bn;
  p.tiles_per_group = p.m_tiles * p.n_tiles;
  p.num_mma_tiles = g.n_mma * p.tiles_per_group;
  p.num_tiles = n * p.tiles_per_group;
  p.gran_k = x.fp8 ? x.gran_k : 0;
  // Mixed tile widths are possible (see below): FP8, token-major operands,
  // kernel N a multiple of both 256 and 224.
  const int mix_pct_env = mixed_tiles_percent();
  const bool mixable = x.fp8 && bn == kNarrowBN && Nk % kWideBN == 0 && g.n_mma > 0 &&
                       mix_pct_env != 0;
  p.chunk = !x.fp8                  ? kBf16Chunk
            : x.d_dtype == DG_BF16    ? (mixable ? kFp8ChunkBf16OutMixed : kFp8ChunkBf16Out)
            : (x.c == x.d)            ? kFp8ChunkInPlace
                                      : kFp8Chunk;
  const char *chunk_env = std::getenv("DG_LANE_CHUNK");
  if (chunk_env != nullptr) {   // tuning override (multiple of 4)
    const int c = std::atoi(chunk_env);
    if (c > 0 && (!x.fp8 || c % 4 == 0)) p.chunk = c;
    else chunk_env = nullptr;
  }
  // Sweep the smaller operand's tiles fastest: the concurrently running tiles
  // then share the larger operand's slices, and the smaller one stays in L2
  // from one sweep to the next.
  p.m_fastest = (Mk <= Nk) ? 1 : 0;
  p.out_mode = (x.d_dtype == DG_BF16) ? OUT_BF16
               : (x.c == nullptr)     ? OUT_F32
               : (x.c == x.d)         ? OUT_F32_REDUCE
                                      : OUT_F32_C;
  p.ks_dev = x.ks_dev;
  // Mixed tile widths (FP8, kernel N a multiple of both 256 and 224): the
  // longest entries are cut into 256-column tiles, which load fewer operand
  // bytes per multiply-add than 224-column ones (12.5 % with token-major
  // operands, whose 128-byte B rows then fill whole 32-byte sectors; 6.7 %
  // with K-major ones).  Only the first
  // accumulator holds 256 columns, so only lane 0 takes wide tiles, and each
  // of its turns on them pairs with a narrow tile of lane 1: entries become
  // wide, longest first, while the narrow tiles left still cover the lane-0
  // turns that the wide ones take.
  // (the share, unless DG_MIXED_TILES sets it: 50 % for FP32 output without
  // an accumulator in place, whose heavy drains favour more narrow tiles,
  // 100 % otherwise; measured)
  const int mix_pct = mix_pct_env >= 0 ? mix_pct_env
                      : (p.out_mode == OUT_F32 || p.out_mode == OUT_F32_C) ? kMixPercentF32
                                                                            : kMixPercent;
  if (mixable) {
    const int ntw = Nk / kWideBN;
    const int64_t tpg_w = static_cast<int64_t>(p.m_tiles) * ntw;
    int64_t narrow = static_cast<int64_t>(n) * tpg;   // narrow tiles with no wide entry
    int64_t turns = 0;                                // lane-0 turns of the wide tiles
    int nw = 0;
    for (; nw < g.n_mma; ++nw) {
      const int64_t nk = (ents[nw].k_len + 127) / 128;
      const int64_t t = tpg_w * ((nk + p.chunk - 1) / p.chunk);
      if ((turns + t) * 100 > (narrow - tpg) * mix_pct) break;
      turns += t;
      narrow -= tpg;
    }
    if (nw > 0) {
      g.bn = kWideBN;
      p.n_wide = nw;
      p.n_tiles_w = ntw;
      p.tpg_w = static_cast<int>(tpg_w);
      p.wide_tiles = static_cast<int>(nw * tpg_w);
      p.num_mma_tiles = p.wide_tiles + (g.n_mma - nw) * tpg;
      p.num_tiles = p.wide_tiles + (n - nw) * tpg;
    } else if (p.chunk == kFp8ChunkBf16OutMixed && chunk_env == nullptr &&
               x.d_dtype == DG_BF16) {
      p.chunk = kFp8ChunkBf16Out;   // no wide entry: the 224-only kernel's chunk
    }
  }
  g.sf_bytes = (x.fp8 && g.n_mma > 0) ? plan_scale_pack(p, pk, g.n_mma, x.gran_k, bn) : 0;
  set_derived(p, n);
}

dg_status grouped_maps(const GroupedArgs &x, const GroupedPlan &g, WgradParams &p) {
  dg_status s = DG_OK;
  const uint64_t M = x.M, N = x.N, G = x.G, SK = x.sum_k;
  const uint64_t MK = p.M, NK = p.N;
  const void *ka = g.trans ? x.b : x.a;
  const void *kb = g.trans ? x.a : x.b;
  const int bn = g.bn;
  if (p.num_mma_tiles > 0) {
    if (x.fp8 && x.kmajor) {
      // K-major: rows of sum_k bytes; one box = 128 tokens x 128 rows (A) or
      // x bn / 2 rows (B), 128-byte swizzled.
      const uint64_t da[2] = {SK, MK}, db[2] = {SK, NK}, st[1] = {SK};
      const uint32_t box[2] = {128, 128};
      const uint32_t boxb[2] = {128, static_cast<uint32_t>(bn / 2)};
      if ((s = encode(&p.tmA, CU_TENSOR_MAP_DATA_TYPE_UINT8, ka, 2, da, st, box,
                      CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, "a")) ||
          (s = encode(&p.tmB, CU_TENSOR_MAP_DATA_TYPE_UINT8, kb, 2, db, st, boxb,
                      CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, "b")))
        return s;
      // mixed widths: the narrow tiles' B boxes
      const uint32_t boxn[2] = {128, static_cast<uint32_t>(kNarrowBN / 2)};
      if (bn == kWideBN &&
          (s = encode(&p.tmBn, CU_TENSOR_MAP_DATA_TYPE_UINT8, kb, 2, db, st, boxn,
                      CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, "b")))
        return s;
    } else if (x.fp8) {
      const uint64_t da[2] = {MK, SK}, sa[1] = {MK};
      const uint64_t db[2] = {NK, SK}, sb[1] = {NK};
      const uint32_t box[2] = {128, 128};
      // B: one box per CTA covers its bn / 2 columns (<= one 128-byte atom);
      // mixed widths: tmB for the wide tiles, tmBn for the narrow ones
      const uint32_t boxb[2] = {static_cast<uint32_t>(std::min(128, bn / 2)), 128};
      const uint32_t boxn[2] = {static_cast<uint32_t>(kNarrowBN / 2), 128};
      if ((s = encode(&p.tmA, CU_TENSOR_MAP_DATA_TYPE_UINT8, ka, 2, da, sa, box,
                      CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, "a")) ||
          (s = encode(&p.tmB, CU_TENSOR_MAP_DATA_TYPE_UINT8, kb, 2, db, sb, boxb,
                      CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, "b")))
        return s;
      if (bn == kWideBN &&
          (s = encode(&p.tmBn, CU_TENSOR_MAP_DATA_TYPE_UINT8, kb, 2, db, sb, boxn,
                      CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, "b")))
        return s;
    } else {
      const uint64_t da[2] = {M, SK}, sa[1] = {2 * M};
      const uint64_t db[2] = {N, SK}, sb[1] = {2 * N};
      const uint32_t box[2] = {64, 64};
      const uint32_t boxb[2] = {static_cast<uint32_t>(std::min(64, bn / 2)), 64};
      if ((s = encode(&p.tmA, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, x.a, 2, da, sa, box,
                      CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, "a")) ||
          (s = encode(&p.tmB, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, x.b, 2, db, sb, boxb,
                      CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, "b")))
        return s;
    }
  }
  const bool bf = (x.d_dtype == DG_BF16);
  const uint64_t es = bf ? 2 : 4;
  const uint64_t dd[3] = {N, M, G}, sd[2] = {es * N, es * N * M};
  const uint32_t box[3] = {kEpiCols, 32, 1};
  if ((s = encode(&p.tmD, bf ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32,
                  x.d, 3, dd, sd, box, epi_swizzle(bf ? 2 : 4), CU_TENSOR_MAP_L2_PROMOTION_NONE,
                  "d")))
    return s;
  if (p.out_mode == OUT_F32_C &&
      (s = encode(&p.tmC, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, x.c, 3, dd, sd, box, epi_swizzle(4),
                  CU_TENSOR_MAP_L2_PROMOTION_NONE, "c")))
    return s;
  return DG_OK;
}

dg_status grouped_scale_maps(const GroupedArgs &x, const GroupedPlan &g, void *scratch,
                             WgradParams &p, PackParams &pk) {
  (void)x;
  bind_scale_pack(pk, scratch, g.ksfa, g.ksfb);
  const uint64_t rec[1] = {512};
  const uint64_t dpa[2] = {128, static_cast<uint64_t>(pk.n_groups) * pk.MC};
  const uint64_t dpb[2] = {128, (static_cast<uint64_t>(pk.GW) * pk.NTW +
                                static_cast<uint64_t>(pk.n_groups - pk.GW) * pk.NT) * pk.CB};
  const uint32_t bpa[2] = {128, 1}, bpb[2] = {128, static_cast<uint32_t>(pk.CB)};
  dg_status s;
  if ((s = encode(&p.tmSFA, CU_TENSOR_MAP_DATA_TYPE_UINT32, pk.sfa_p, 2, dpa, rec, bpa,
                  CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_NONE, "sfa records")) ||
      (s = encode(&p.tmSFB, CU_TENSOR_MAP_DATA_TYPE_UINT32, pk.sfb_p, 2, dpb, rec, bpb,
                  CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_NONE, "sfb records")))
    return s;
  return DG_OK;
}

cudaError_t grouped_launch(const GroupedArgs &x, const GroupedPlan &g, WgradParams &p, int sms) {
  const int pairs = std::min(sms / 2, p.num_tiles);
  return !x.fp8               ? launch_kgrouped_bf16(p, g.bn, pairs, x.stream)
         : x.kmajor && g.trans ? launch_kgrouped_fp8_nt_t(p, g.bn, pairs, x.stream)
         : x.kmajor           ? launch_kgrouped_fp8_nt(p, g.bn, pairs, x.stream)
         : g.trans            ? launch_kgrouped_fp8_t(p, g.bn, pairs, x.stream)
                              : launch_kgrouped_fp8(p, g.bn, pairs, x.stream);
}

}  // namespace dg

namespace {

using dg::GroupedArgs;
using dg::wait_limit_ns;

dg_status run_grouped(const GroupedArgs &x) {
  const char *fn = x.fn;
  dg_status s = dg::grouped_validate(x);
  if (s != DG_OK) return s;
  if (x.G == 0) return ok();
  DeviceState *dev = nullptr;
  if ((s = device_state(&dev)) != DG_OK) return s;

  // ---- schedule: longest entries first, then output-only (fill) experts
  // ~29 KB and ~12 KB: per-thread storage rather than the stack or the heap
  static thread_local dg::WgradParams t_p;
  static thread_local dg::PackParams t_pk;
  dg::WgradParams &p = t_p;
  dg::PackParams &pk = t_pk;
  dg::GroupedPlan g{};
  dg::grouped_schedule(x, dev->sms, p, pk, g);
  p.wait_limit_ns = wait_limit_ns();
  p.status = dev->status;
#ifdef DG_KERNEL_TIMERS
  p.timers = g_timers;
#endif
  if (log_enabled()) {
    int empty = 0, max_k = 0;
    for (int e = 0; e < x.G; ++e) {
      empty += (x.ks_host[e] == 0);
      max_k = std::max(max_k, x.ks_host[e]);
    }
    std::fprintf(stderr,
                 "[dg] %s: G=%d M=%d N=%d sum_k=%lld (%d empty, max K %d) | %s operands, %s tiles "
                 "256 x %d, %d x %d per expert (%d entries of 256 x 256 tiles, %d x %d) | "
                 "%d GEMM entries (+%d from splits along K), "
                 "%d GEMM tiles + %d output-only | out=%s | pairs=%d\n",
                 fn, x.G, x.M, x.N, static_cast<long long>(x.sum_k), empty, max_k,
                 x.kmajor ? "K-major" : "token-major", g.trans ? "transposed" : "direct",
                 g.bn == dg::kWideBN ? dg::kNarrowBN : g.bn, p.m_tiles, p.n_tiles, p.n_wide,
                 p.m_tiles, p.n_tiles_w, g.n_mma, g.n_mma - (x.G - empty), p.num_mma_tiles,
                 p.num_tiles - p.num_mma_tiles,
                 p.out_mode == dg::OUT_BF16        ? "bf16"
                 : p.out_mode == dg::OUT_F32       ? "f32"
                 : p.out_mode == dg::OUT_F32_REDUCE ? "f32 += (reduce-add)"
                                                    : "f32 = C +",
                 std::min(dev->sms / 2, p.num_tiles));
  }
  if (p.num_tiles == 0) return ok();     // every expert empty and D accumulates in place
  if ((s = dg::grouped_maps(x, g, p)) != DG_OK) return s;

  // ---- FP8 scale records: scratch from the pool, their tensor maps, the pack pass
  void *scratch = nullptr;
  cudaError_t e = cudaSuccess;
  if (g.sf_bytes > 0) {
    if ((e = cudaMallocFromPoolAsync(&scratch, g.sf_bytes, dev->pool, x.stream)) != cudaSuccess)
      return fail(DG_ERR_CUDA, "%s: scale scratch (%zu bytes): %s", fn, g.sf_bytes,
                  cudaGetErrorString(e));
    if ((s = dg::grouped_scale_maps(x, g, scratch, p, pk)) != DG_OK) {
      cudaFreeAsync(scratch, x.stream);
      return s;
    }
    if ((e = dg::launch_pack_scales(pk, x.stream)) != cudaSuccess) {
      cudaFreeAsync(scratch, x.stream);
      return fail(DG_ERR_CUDA, "%s: scale pack launch failed: %s", fn, cudaGetErrorString(e));
    }
    p.pdl = dg::pdl_requested() ? 1 : 0;   // the GEMM may start beside the pack pass
  }

  // ---- launch: one persistent CTA pair per two SMs (or per tile when fewer)
  e = dg::grouped_launch(x, g, p, dev->sms);
  if (scratch != nullptr) cudaFreeAsync(scratch, x.stream);   // after the GEMM in stream order
  if (e != cudaSuccess)
    return fail(DG_ERR_CUDA, "%s: launch failed: %s", fn, cudaGetErrorString(e));
  return ok();
}

// M-grouped FP8 data gradient: validation, schedule (one entry per expert with
// tokens), tensor maps, the two scale-pack passes and the GEMM launch.
dg_status run_mgrouped(const void *a, const uint8_t *sfa, const void *w, const uint8_t *sfw,
                       void *d, dg_dtype d_dtype, int G, int K, int N, int64_t sum_m,
                       const int *ms_host, const int *ms_dev, int gran_k, cudaStream_t stream,
                       bool w_kmajor) {
  const char *fn = w_kmajor ? "dg_m_grouped_fp8_dgrad_nt" : "dg_m_grouped_fp8_dgrad";
  if (G < 0) return fail(DG_ERR_INVALID_ARG, "%s: G = %d < 0", fn, G);
  if (G > DG_MAX_GROUPS) return fail(DG_ERR_UNSUPPORTED, "%s: G = %d above DG_MAX_GROUPS", fn, G);
  if (K <= 0 || K % 128)
    return fail(DG_ERR_INVALID_ARG, "%s: K = %d must be a positive multiple of 128", fn, K);
  if (N <= 0 || N % 16)
    return fail(DG_ERR_INVALID_ARG, "%s: N = %d must be a positive multiple of 16", fn, N);
  if (gran_k != 32 && gran_k != 128)
    return fail(DG_ERR_INVALID_ARG, "%s: gran_k = %d (must be 32 or 128)", fn, gran_k);
  if (d_dtype != DG_F32 && d_dtype != DG_BF16)
    return fail(DG_ERR_INVALID_ARG, "%s: unknown output dtype %d", fn, (int)d_dtype);
  if (sum_m < 0) return fail(DG_ERR_INVALID_ARG, "%s: sum_m < 0", fn);
  if (sum_m > (int64_t)0x7FFFFF00)
    return fail(DG_ERR_UNSUPPORTED, "%s: sum_m above 2^31 - 256", fn);
  if (static_cast<int64_t>(G) * K > 0x7FFFFFFFll || static_cast<int64_t>(G) * N > 0x7FFFFFFFll)
    return fail(DG_ERR_UNSUPPORTED, "%s: G * K or G * N above 2^31 - 1", fn);
  if (G == 0) {
    if (sum_m != 0) return fail(DG_ERR_INVALID_ARG, "%s: G = 0 but sum_m = %lld", fn, (long long)sum_m);
    return ok();
  }
  if (ms_host == nullptr || ms_dev == nullptr)
    return fail(DG_ERR_INVALID_ARG, "%s: ms_host and ms_dev are required", fn);
  int64_t total = 0;
  for (int e = 0; e < G; ++e) {
    const int m = ms_host[e];
    if (m < 0) return fail(DG_ERR_INVALID_ARG, "%s: ms[%d] = %d < 0", fn, e, m);
    if (m % 128) return fail(DG_ERR_INVALID_ARG, "%s: ms[%d] = %d is not a multiple of 128", fn, e, m);
    total += m;
  }
  if (total != sum_m)
    return fail(DG_ERR_INVALID_ARG, "%s: sum of ms (%lld) != sum_m (%lld)", fn, (long long)total,
                (long long)sum_m);
  if (sum_m == 0) return ok();
  if (a == nullptr || w == nullptr || d == nullptr || sfa == nullptr || sfw == nullptr ||
      !aligned16(a) || !aligned16(w) || !aligned16(d) || !aligned16(sfa) || !aligned16(sfw))
    return fail(DG_ERR_INVALID_ARG, "%s: a, sfa, w, sfw and d must be 16-byte aligned device pointers",
                fn);
  const int es = (d_dtype == DG_BF16) ? 2 : 4;
  if (static_cast<double>(sum_m) * N * es >= 1099511627776.0)
    return fail(DG_ERR_UNSUPPORTED, "%s: output of 2^40 bytes or more", fn);
  DeviceState *dev = nullptr;
  dg_status s = device_state(&dev);
  if (s != DG_OK) return s;

  const int bn = dg::fp8_pick_block_n(N);
  const int n_tiles = (N + bn - 1) / bn;
  const int KB = K / gran_k;                          // scale columns of A, scale rows per W_e
  const int gs = (gran_k == 128) ? 4 : 1;             // 128-wide k-blocks per scale group
  const int NGK = (K / 128 + gs - 1) / gs;            // scale groups along K
  const int TC = static_cast<int>(sum_m / 128) + 1;   // 128-token chunks (+1: a last odd half)

  std::unique_ptr<dg::WgradParams> hold(new dg::WgradParams);
  dg::WgradParams &p = *hold;
  std::memset(&p, 0, sizeof(p));
  int n_ent = 0;
  int64_t tiles = 0, row = 0;
  for (int e = 0; e < G; ++e) {
    const int m = ms_host[e];
    if (m > 0) {
      dg::SchedEntry &se = p.sched[n_ent];
      se.expert = e;
      se.k_off = w_kmajor ? e * N : e * K;   // the expert's first row of W
      se.k_len = K;
      se.g_off = n_ent * NGK;
      se.k_exp = m;
      se.row_off = static_cast<int>(row);
      se.tile_off = static_cast<int>(tiles);
      tiles += static_cast<int64_t>((m + dg::kPairM - 1) / dg::kPairM) * n_tiles;
      ++n_ent;
    }
    row += m;
  }
  if (tiles > 0x7FFFFFFFll) return fail(DG_ERR_UNSUPPORTED, "%s: more than 2^31 - 1 tiles", fn);
  p.M = K;
  p.N = N;
  p.G = G;
  p.m_tiles = 1;
  p.n_tiles = n_tiles;
  p.tiles_per_group = n_tiles;
  p.num_mma_tiles = static_cast<int>(tiles);
  p.num_tiles = static_cast<int>(tiles);
  p.gran_k = gran_k;
  p.chunk = dg::kFp8Chunk;
  p.out_mode = (d_dtype == DG_BF16) ? dg::OUT_BF16 : dg::OUT_F32;
  p.sf_mc = TC;
  p.mgroup = 1;
  p.n_entries = n_ent;
  p.wait_limit_ns = wait_limit_ns();
  p.status = dev->status;
  p.ks_dev = ms_dev;
#ifdef DG_KERNEL_TIMERS
  p.timers = g_timers;
#endif
  if (log_enabled())
    std::fprintf(stderr,
                 "[dg] %s: G=%d K=%d N=%d sum_m=%lld | %d experts with tokens, tiles 256 x %d, "
                 "%lld tiles | out=%s | pairs=%d\n",
                 fn, G, K, N, static_cast<long long>(sum_m), n_ent, bn,
                 static_cast<long long>(tiles), d_dtype == DG_BF16 ? "bf16" : "f32",
                 std::min<int64_t>(dev->sms / 2, tiles) > 0 ? static_cast<int>(std::min<int64_t>(dev->sms / 2, tiles)) : 0);

  // ---- tensor maps: dy as {K, sum_m} (K-major boxes of 128 x 128), the
  // weights as {N, G K} (MN-major boxes of bn / 2 x 128), D as {N, sum_m, 1}
  const uint64_t SM = static_cast<uint64_t>(sum_m), UK = K, UN = N, GK = static_cast<uint64_t>(G) * K;
  const uint64_t GN = static_cast<uint64_t>(G) * N;
  {
    const uint64_t da[2] = {UK, SM}, sa[1] = {UK};
    // W [G, K, N] as {N, G K} with boxes of bn / 2 x 128 rows; K-major W
    // [G, N, K] as {K, G N} with boxes of 128 bytes of K x bn / 2 rows
    const uint64_t db[2] = {w_kmajor ? UK : UN, w_kmajor ? GN : GK};
    const uint64_t sb[1] = {w_kmajor ? UK : UN};
    const uint32_t boxa[2] = {128, 128};
    const uint32_t boxb[2] = {w_kmajor ? 128u : static_cast<uint32_t>(std::min(128, bn / 2)),
                              w_kmajor ? static_cast<uint32_t>(bn / 2) : 128u};
    if ((s = encode(&p.tmA, CU_TENSOR_MAP_DATA_TYPE_UINT8, a, 2, da, sa, boxa,
                    CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, "a")) ||
        (s = encode(&p.tmB, CU_TENSOR_MAP_DATA_TYPE_UINT8, w, 2, db, sb, boxb,
                    CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, "w")))
      return s;
    const bool bf = (d_dtype == DG_BF16);
    const uint64_t dd[3] = {UN, SM, 1}, sd[2] = {es * UN, es * UN * SM};
    const uint32_t box[3] = {dg::kEpiCols, 32, 1};
    if ((s = encode(&p.tmD, bf ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32,
                    d, 3, dd, sd, box, dg::epi_swizzle(es), CU_TENSOR_MAP_L2_PROMOTION_NONE, "d")))
      return s;
  }

  // ---- scale records: A per token chunk ([NGK][TC]), W per (entry, group, N tile)
  std::unique_ptr<dg::PackParams> pk_hold(new dg::PackParams);
  dg::PackParams &pk = *pk_hold;
  std::memset(&pk, 0, sizeof(pk));
  for (int i = 0; i < n_ent; ++i) {
    pk.g_off[i] = p.sched[i].g_off;
    pk.row_off[i] = p.sched[i].expert * KB;
    pk.row_end[i] = pk.row_off[i] + KB;
  }
  pk.M = 0;
  pk.N = N;
  pk.MC = 0;
  pk.NT = n_tiles;
  pk.CB = (bn + 127) / 128;
  pk.BN = bn;
  pk.n_entries = n_ent;
  pk.n_groups = n_ent * NGK;
  const size_t a_rec = static_cast<size_t>(NGK) * TC * 512;
  const size_t b_rec = static_cast<size_t>(pk.n_groups) * pk.NT * pk.CB * 512;
  void *scratch = nullptr;
  cudaError_t e = cudaMallocFromPoolAsync(&scratch, a_rec + b_rec, dev->pool, stream);
  if (e != cudaSuccess)
    return fail(DG_ERR_CUDA, "%s: scale scratch (%zu bytes): %s", fn, a_rec + b_rec,
                cudaGetErrorString(e));
  dg::TokenPackParams tp;
  tp.sfa = sfa;
  tp.sfa_p = static_cast<uint32_t *>(scratch);
  tp.sum_m = sum_m;
  tp.KB = KB;
  tp.NGK = NGK;
  tp.TC = TC;
  pk.sfa = nullptr;
  pk.sfb = sfw;
  pk.sfa_p = nullptr;
  pk.sfb_p = reinterpret_cast<uint32_t *>(static_cast<uint8_t *>(scratch) + a_rec);
  {
    const uint64_t rec[1] = {512};
    const uint64_t dpa[2] = {128, static_cast<uint64_t>(NGK) * TC};
    const uint64_t dpb[2] = {128, static_cast<uint64_t>(pk.n_groups) * pk.NT * pk.CB};
    const uint32_t bpa[2] = {128, 1}, bpb[2] = {128, static_cast<uint32_t>(pk.CB)};
    if ((s = encode(&p.tmSFA, CU_TENSOR_MAP_DATA_TYPE_UINT32, tp.sfa_p, 2, dpa, rec, bpa,
                    CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_NONE, "sfa records")) ||
        (s = encode(&p.tmSFB, CU_TENSOR_MAP_DATA_TYPE_UINT32, pk.sfb_p, 2, dpb, rec, bpb,
                    CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_NONE, "sfw records"))) {
      cudaFreeAsync(scratch, stream);
      return s;
    }
  }
  if ((e = dg::launch_pack_token_scales(tp, stream)) != cudaSuccess ||
      (e = dg::launch_pack_scales(pk, stream)) != cudaSuccess) {
    cudaFreeAsync(scratch, stream);
    return fail(DG_ERR_CUDA, "%s: scale pack launch failed: %s", fn, cudaGetErrorString(e));
  }
  dg::set_derived(p, n_ent);
  p.pdl = dg::pdl_requested() ? 1 : 0;   // the GEMM may start beside the second pack pass
  const int pairs = static_cast<int>(std::min<int64_t>(dev->sms / 2, tiles));
  e = w_kmajor ? dg::launch_mgrouped_fp8_nt(p, bn, pairs, stream)
               : dg::launch_mgrouped_fp8(p, bn, pairs, stream);
  cudaFreeAsync(scratch, stream);   // after the GEMM in stream order
  if (e != cudaSuccess) return fail(DG_ERR_CUDA, "%s: launch failed: %s", fn, cudaGetErrorString(e));
  return ok();
}

dg::CastArgs cast_args(const void *x, const uint8_t *x_sf, const int *src_rows, int64_t T_src,
                       int64_t T, int C, void *q, uint8_t *sf) {
  dg::CastArgs a;
  std::memset(&a, 0, sizeof(a));
  a.x = x;
  a.x_sf = x_sf;
  a.src_rows = src_rows;
  a.T_src = T_src;
  a.T = T;
  a.C = C;
  a.q = static_cast<uint8_t *>(q);
  a.sf = sf;
  return a;
}

// Validation and launch shared by the three column-block casts.  a.x_sf set:
// E4M3 source with 1 x 128 scales (C a multiple of 128); a.src_rows set: MoE
// layout gather from T_src source rows.
dg_status run_cast(const char *fn, dg::CastArgs a, dg_layout q_layout, int gran_k,
                   cudaStream_t stream) {
  const bool fp8 = (a.x_sf != nullptr);
  if (gran_k != 32 && gran_k != 128)
    return fail(DG_ERR_INVALID_ARG, "%s: gran_k = %d (must be 32 or 128)", fn, gran_k);
  if (q_layout != DG_TOKEN_MAJOR && q_layout != DG_CHANNEL_MAJOR)
    return fail(DG_ERR_INVALID_ARG, "%s: unknown layout %d", fn, (int)q_layout);
  if (a.T < 0 || a.T % gran_k)
    return fail(DG_ERR_INVALID_ARG, "%s: T = %lld must be a non-negative multiple of gran_k",
                fn, (long long)a.T);
  const int cmult = fp8 ? 128 : 16;
  if (a.C <= 0 || a.C % cmult)
    return fail(DG_ERR_INVALID_ARG, "%s: C = %d must be a positive multiple of %d", fn, a.C,
                cmult);
  if ((a.C + 255) / 256 > 65535) return fail(DG_ERR_UNSUPPORTED, "%s: C too large", fn);
  if ((a.T + 127) / 128 > 0x7FFFFFFFll) return fail(DG_ERR_UNSUPPORTED, "%s: T too large", fn);
  if (a.src_rows != nullptr && a.T_src > 0x7FFFFFFFll)
    return fail(DG_ERR_UNSUPPORTED, "%s: T_src above 2^31 - 1 (int32 row indices)", fn);
  if (a.T == 0) return ok();
  const bool need_x = (a.src_rows == nullptr) || a.T_src > 0;
  if ((need_x && (a.x == nullptr || !aligned16(a.x))) || a.q == nullptr || a.sf == nullptr ||
      !aligned16(a.q) || !aligned16(a.sf) || (fp8 && need_x && !aligned16(a.x_sf)) ||
      (a.src_rows != nullptr && !aligned16(a.src_rows)))
    return fail(DG_ERR_INVALID_ARG, "%s: device pointers must be non-NULL and 16-byte aligned",
                fn);
  DeviceState *dev = nullptr;
  dg_status s = device_state(&dev);
  if (s != DG_OK) return s;
  a.status = dev->status;
  a.wait_limit_ns = wait_limit_ns();
  // BF16 rows gathered into the token-major layout: the rows come in by TMA
  // (four indexed rows per instruction) through a map of x as {C, T_src}.
  if (!fp8 && a.src_rows != nullptr && q_layout == DG_TOKEN_MAJOR && a.T_src > 0) {
    const uint64_t dims[2] = {static_cast<uint64_t>(a.C), static_cast<uint64_t>(a.T_src)};
    const uint64_t strides[1] = {static_cast<uint64_t>(a.C) * 2};
    const uint32_t box[2] = {256, 1};
    if ((s = encode(&a.tmx, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, a.x, 2, dims, strides, box,
                    CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_128B, "x rows")))
      return s;
    a.use_tmx = 1;
  }
  cudaError_t e = dg::launch_cast_colblock(a, q_layout == DG_CHANNEL_MAJOR, gran_k, stream);
  if (e != cudaSuccess)
    return fail(DG_ERR_CUDA, "%s: launch failed: %s", fn, cudaGetErrorString(e));
  return ok();
}

}  // namespace

extern "C" {

dg_status dg_k_grouped_fp8_wgrad(const void *a, const uint8_t *sfa, const void *b,
                                 const uint8_t *sfb, void *d, dg_dtype d_dtype, const float *c,
                                 int G, int M, int N, int64_t sum_k, const int *ks_host,
                                 const int *ks_dev, int gran_k, dg_stream_t stream) {
  GroupedArgs x{"dg_k_grouped_fp8_wgrad", true, false, a, b, sfa, sfb, d, d_dtype, c, G, M, N,
                sum_k, ks_host, ks_dev, gran_k, reinterpret_cast<cudaStream_t>(stream)};
  return run_grouped(x);
}

dg_status dg_k_grouped_fp8_wgrad_nt(const void *a, const uint8_t *sfa, const void *b,
                                    const uint8_t *sfb, void *d, dg_dtype d_dtype,
                                    const float *c, int G, int M, int N, int64_t sum_k,
                                    const int *ks_host, const int *ks_dev, int gran_k,
                                    dg_stream_t stream) {
  GroupedArgs x{"dg_k_grouped_fp8_wgrad_nt", true, true, a, b, sfa, sfb, d, d_dtype, c, G, M,
                N, sum_k, ks_host, ks_dev, gran_k, reinterpret_cast<cudaStream_t>(stream)};
  return run_grouped(x);
}

dg_status dg_k_grouped_bf16_wgrad(const void *a, const void *b, void *d, dg_dtype d_dtype,
                                  const float *c, int G, int M, int N, int64_t sum_k,
                                  const int *ks_host, const int *ks_dev, dg_stream_t stream) {
  GroupedArgs x{"dg_k_grouped_bf16_wgrad", false, false, a, b, nullptr, nullptr, d, d_dtype, c,
                G, M, N, sum_k, ks_host, ks_dev, 0, reinterpret_cast<cudaStream_t>(stream)};
  return run_grouped(x);
}

dg_status dg_m_grouped_fp8_dgrad(const void *a, const uint8_t *sfa, const void *w,
                                 const uint8_t *sfw, void *d, dg_dtype d_dtype, int G, int K,
                                 int N, int64_t sum_m, const int *ms_host, const int *ms_dev,
                                 int gran_k, dg_stream_t stream) {
  return run_mgrouped(a, sfa, w, sfw, d, d_dtype, G, K, N, sum_m, ms_host, ms_dev, gran_k,
                      reinterpret_cast<cudaStream_t>(stream), false);
}

dg_status dg_m_grouped_fp8_dgrad_nt(const void *a, const uint8_t *sfa, const void *w,
                                    const uint8_t *sfw, void *d, dg_dtype d_dtype, int G, int K,
                                    int N, int64_t sum_m, const int *ms_host, const int *ms_dev,
                                    int gran_k, dg_stream_t stream) {
  return run_mgrouped(a, sfa, w, sfw, d, d_dtype, G, K, N, sum_m, ms_host, ms_dev, gran_k,
                      reinterpret_cast<cudaStream_t>(stream), true);
}

dg_status dg_quant_transpose_fp8(const void *x, int64_t T, int C, void *q, uint8_t *sf,
                                 dg_layout q_layout, int gran_k, dg_stream_t stream) {
  dg::CastArgs a = cast_args(x, nullptr, nullptr, T, T, C, q, sf);
  return run_cast("dg_quant_transpose_fp8", a, q_layout, gran_k,
                  reinterpret_cast<cudaStream_t>(stream));
}

dg_status dg_requant_transpose_fp8(const void *q_in, const uint8_t *sf_in, int64_t T, int C,
                                   void *q, uint8_t *sf, dg_layout q_layout, int gran_k,
                                   dg_stream_t stream) {
  const char *fn = "dg_requant_transpose_fp8";
  if (T > 0 && sf_in == nullptr)
    return fail(DG_ERR_INVALID_ARG, "%s: sf_in is required", fn);
  dg::CastArgs a = cast_args(q_in, sf_in, nullptr, T, T, C, q, sf);
  return run_cast(fn, a, q_layout, gran_k, reinterpret_cast<cudaStream_t>(stream));
}

dg_status dg_quant_moe_layout_fp8(const void *x, const uint8_t *x_sf, int64_t T_src, int C,
                                  const int *src_rows, int64_t T, void *q, uint8_t *sf,
                                  dg_layout q_layout, int gran_k, dg_stream_t stream) {
  const char *fn = "dg_quant_moe_layout_fp8";
  if (T_src < 0) return fail(DG_ERR_INVALID_ARG, "%s: T_src < 0", fn);
  if (T > 0 && src_rows == nullptr)
    return fail(DG_ERR_INVALID_ARG, "%s: src_rows is required", fn);
  dg::CastArgs a = cast_args(x, x_sf, src_rows, T_src, T, C, q, sf);
  return run_cast(fn, a, q_layout, gran_k, reinterpret_cast<cudaStream_t>(stream));
}

dg_status dg_moe_layout_plan(const int *topk_idx, int64_t T_tok, int topk, int G, int align,
                             int *ks, int *src_rows, int *pair_rows, int64_t cap,
                             dg_stream_t stream) {
  const char *fn = "dg_moe_layout_plan";
  if (T_tok < 0 || topk < 1)
    return fail(DG_ERR_INVALID_ARG, "%s: T_tok = %lld, topk = %d", fn, (long long)T_tok, topk);
  if (G < 1 || G > DG_MAX_GROUPS)
    return fail(G < 1 ? DG_ERR_INVALID_ARG : DG_ERR_UNSUPPORTED, "%s: G = %d (1..%d)", fn, G,
                DG_MAX_GROUPS);
  if (align < 1 || align > 65536)
    return fail(DG_ERR_INVALID_ARG, "%s: align = %d (1..65536)", fn, align);
  const int64_t n = T_tok * static_cast<int64_t>(topk);
  const int64_t need = n + static_cast<int64_t>(G) * (align - 1);
  if (T_tok > 0x7FFFFFFFll || need > 0x7FFFFFFFll)
    return fail(DG_ERR_UNSUPPORTED, "%s: layout rows above 2^31 - 1", fn);
  if (cap < need)
    return fail(DG_ERR_INVALID_ARG, "%s: cap = %lld < T_tok * topk + G * (align - 1) = %lld",
                fn, (long long)cap, (long long)need);
  if (ks == nullptr || src_rows == nullptr || !aligned16(ks) || !aligned16(src_rows) ||
      (n > 0 && (topk_idx == nullptr || !aligned16(topk_idx))) ||
      (pair_rows != nullptr && !aligned16(pair_rows)))
    return fail(DG_ERR_INVALID_ARG, "%s: device pointers must be non-NULL and 16-byte aligned",
                fn);
  DeviceState *dev = nullptr;
  dg_status s = device_state(&dev);
  if (s != DG_OK) return s;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  void *scratch = nullptr;
  cudaError_t e =
      cudaMallocFromPoolAsync(&scratch, dg::moe_plan_scratch_bytes(n, G), dev->pool, st);
  if (e != cudaSuccess)
    return fail(DG_ERR_CUDA, "%s: scratch: %s", fn, cudaGetErrorString(e));
  dg::MoePlanArgs a{topk_idx, n, topk, G, align, ks, src_rows, pair_rows, cap, scratch,
                    dev->status};
  e = dg::launch_moe_layout_plan(a, dev->sms, st);
  cudaFreeAsync(scratch, st);   // after the plan's kernels in stream order
  if (e != cudaSuccess)
    return fail(DG_ERR_CUDA, "%s: launch failed: %s", fn, cudaGetErrorString(e));
  return ok();
}

dg_status dg_swiglu_backward_quant_fp8(const void *h, const void *da, int64_t T, int I,
                                       void *q_dh, uint8_t *sf_dh, void *q_a, uint8_t *sf_a,
                                       int gran_k, dg_stream_t stream) {
  const char *fn = "dg_swiglu_backward_quant_fp8";
  if (gran_k != 32 && gran_k != 128)
    return fail(DG_ERR_INVALID_ARG, "%s: gran_k = %d (must be 32 or 128)", fn, gran_k);
  if (T < 0 || T % gran_k)
    return fail(DG_ERR_INVALID_ARG, "%s: T = %lld must be a non-negative multiple of gran_k",
                fn, (long long)T);
  if (I <= 0 || I % 16)
    return fail(DG_ERR_INVALID_ARG, "%s: I = %d must be a positive multiple of 16", fn, I);
  if ((q_a == nullptr) != (sf_a == nullptr))
    return fail(DG_ERR_INVALID_ARG, "%s: q_a and sf_a go together", fn);
  if ((I + 127) / 128 > 65535 || ((T + 127) / 128) * ((I + 31) / 32) > 0x7FFFFFFFll)
    return fail(DG_ERR_UNSUPPORTED, "%s: T or I too large", fn);
  if (T == 0) return ok();
  if (h == nullptr || da == nullptr || q_dh == nullptr || sf_dh == nullptr || !aligned16(h) ||
      !aligned16(da) || !aligned16(q_dh) || !aligned16(sf_dh) ||
      (q_a != nullptr && (!aligned16(q_a) || !aligned16(sf_a))))
    return fail(DG_ERR_INVALID_ARG, "%s: device pointers must be non-NULL and 16-byte aligned",
                fn);
  DeviceState *dev = nullptr;
  dg_status s = device_state(&dev);
  if (s != DG_OK) return s;
  static thread_local dg::SwigluArgs a;
  std::memset(&a, 0, sizeof(a));
  // h as {2I, T} and da as {I, T}, BF16, boxes of 32 channels x 128 tokens
  const uint64_t dh[2] = {2 * static_cast<uint64_t>(I), static_cast<uint64_t>(T)};
  const uint64_t sh[1] = {4 * static_cast<uint64_t>(I)};
  const uint64_t dd[2] = {static_cast<uint64_t>(I), static_cast<uint64_t>(T)};
  const uint64_t sd[1] = {2 * static_cast<uint64_t>(I)};
  const uint32_t box[2] = {32, 128};
  if ((s = encode(&a.tm_h, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, h, 2, dh, sh, box,
                  CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_128B, "h")) ||
      (s = encode(&a.tm_da, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, da, 2, dd, sd, box,
                  CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_128B, "da")))
    return s;
  a.T = T;
  a.I = I;
  a.n_tt = static_cast<int>((T + 127) / 128);
  a.n_tc = (I + 31) / 32;
  a.q_dh = static_cast<uint8_t *>(q_dh);
  a.sf_dh = sf_dh;
  a.q_a = static_cast<uint8_t *>(q_a);
  a.sf_a = sf_a;
  a.status = dev->status;
  a.wait_limit_ns = dg::wait_limit_ns();
  cudaError_t e = dg::launch_swiglu_bwd_cast(a, gran_k, 2 * dev->sms,
                                             reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess)
    return fail(DG_ERR_CUDA, "%s: launch failed: %s", fn, cudaGetErrorString(e));
  return ok();
}

const char *dg_last_error(void) { return g_err.c_str(); }

dg_status dg_sync_check(dg_stream_t stream) {
  // Reads the records that exist; allocates nothing (a device on which no
  // allocating entry point has run has no ordinary record yet).
  int devi = 0;
  cudaError_t e = cudaGetDevice(&devi);
  if (e != cudaSuccess) return fail(DG_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
  dg::DevStatus *rec = nullptr;
  if (devi >= 0 && devi < kMaxDevices) {
    std::lock_guard<std::mutex> lock(g_mu);
    if (g_dev[devi].init) {
      if (!g_dev[devi].arch_ok)
        return fail(DG_ERR_UNSUPPORTED, "device is sm_%d%d; this library is built for sm_103a only",
                    g_dev[devi].major, g_dev[devi].minor);
      rec = g_dev[devi].status;
    }
  }
  e = cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return fail(DG_ERR_CUDA, "stream synchronise: %s", cudaGetErrorString(e));
  dg::DevStatus st{};
  if (rec != nullptr) {
    if ((e = cudaMemcpy(&st, rec, sizeof(st), cudaMemcpyDeviceToHost)) != cudaSuccess)
      return fail(DG_ERR_CUDA, "status read: %s", cudaGetErrorString(e));
    if (st.code != dg::DEV_OK && (e = cudaMemset(rec, 0, sizeof(st))) != cudaSuccess)
      return fail(DG_ERR_CUDA, "status reset: %s", cudaGetErrorString(e));
  }
  // The allocation-free entry point's record (read and cleared likewise).
  dg::DevStatus na{};
  bool present = false;
  if ((e = dg::noalloc_take_status(&na, &present)) != cudaSuccess)
    return fail(DG_ERR_CUDA, "status read: %s", cudaGetErrorString(e));
  if (st.code == dg::DEV_OK && present) st = na;
  if (st.code == dg::DEV_OK) return ok();
  if (st.code == dg::DEV_TIMEOUT)
    return fail(DG_ERR_TIMEOUT, "device wait timed out (site 0x%x, block %d, detail %d)",
                st.where, st.block, st.detail);
  if (st.code == dg::DEV_BAD_ROW)
    return fail(DG_ERR_INVALID_ARG, "a src_rows entry lies outside [-1, T_src)");
  if (st.code == dg::DEV_BAD_ROUTE)
    return fail(DG_ERR_INVALID_ARG, "a topk_idx entry lies outside [-1, G)");
  return fail(DG_ERR_INVALID_ARG, "ks_dev does not match ks_host");
}

int dg_version(void) { return 100; }

}  // extern "C"
