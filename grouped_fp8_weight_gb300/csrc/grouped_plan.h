// Host-side steps of a K-grouped weight-gradient call, shared by the ordinary
// entry points (api.cu) and the allocation-free FP8 one (noalloc.cu), so that
// both validate, schedule and encode a problem identically and differ only in
// where the status record and the packed scale records live.
#pragma once

#include <cstddef>
#include <cstdint>

#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include "dg_wgrad.h"
#include "wgrad_params.h"

namespace dg {

// Records a formatted message for dg_last_error and returns s.
dg_status failf(dg_status s, const char *fmt, ...);
void set_last_error(const char *msg);

// cuTensorMapEncodeTiled, resolved once per process (no allocation); null if
// the driver does not provide it.
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder();

// Bounded-wait limit of every kernel wait, from DG_WAIT_LIMIT_US or
// DG_WAIT_LIMIT_MS (read at each call; default 4 s).
uint64_t wait_limit_ns();

// DG_DETERMINISTIC set (and not "0") in the environment, read at each call:
// in-place accumulation keeps every expert in one schedule entry (no split
// along K), so every element of D is added to once and the result is bitwise
// reproducible, at some cost in balance when one expert holds most tokens.
bool deterministic_requested();

// DG_PDL=0 in the environment (read at each call) launches an FP8 GEMM only
// after its scale-pack pass has completed, instead of as a programmatic
// dependent that starts beside it.
bool pdl_requested();

struct GroupedArgs {
  const char *fn;   // entry-point name for messages
  bool fp8;
  bool kmajor;      // FP8 only: a [M, sum_k], b [N, sum_k] (NT) instead of [sum_k, M], [sum_k, N]
  const void *a, *b;
  const uint8_t *sfa, *sfb;
  void *d;
  dg_dtype d_dtype;
  const float *c;
  int G, M, N;
  int64_t sum_k;
  const int *ks_host, *ks_dev;
  int gran_k;
  cudaStream_t stream;
};

// What the schedule decided, in the kernel's orientation.
struct GroupedPlan {
  bool trans;          // D^T tiles: the kernel's A is the caller's b
  int bn;              // tile width
  int n_sched;         // schedule entries (GEMM entries first, then output-only)
  int n_mma;           // GEMM entries
  size_t sf_bytes;     // packed scale-record bytes (FP8; 0 without GEMM work)
  const uint8_t *ksfa, *ksfb;   // scales in the kernel's roles
};

// Argument checks (no CUDA call; nothing is enqueued on failure).
dg_status grouped_validate(const GroupedArgs &x);

// Schedule (longest entries first, output-only experts last; in-place
// accumulation splits experts longer than a quarter of a CTA pair's fair share
// along K when sms > 0, unless deterministic_requested()), tile counts, output
// mode and the scale-pack plan into p and pk.  No CUDA call.  p.status,
// p.wait_limit_ns and the tensor maps are left to the caller.
void grouped_schedule(const GroupedArgs &x, int sms, WgradParams &p, PackParams &pk,
                      GroupedPlan &g);

// Tensor maps of the operands (in the kernel's roles), D and C.
dg_status grouped_maps(const GroupedArgs &x, const GroupedPlan &g, WgradParams &p);

// Points the scale pack at `scratch` (g.sf_bytes, 16-byte aligned) and
// encodes the two record maps.
dg_status grouped_scale_maps(const GroupedArgs &x, const GroupedPlan &g, void *scratch,
                             WgradParams &p, PackParams &pk);

// The GEMM launch for the plan's variant (one persistent CTA pair per two SMs,
// or per tile when fewer).
cudaError_t grouped_launch(const GroupedArgs &x, const GroupedPlan &g, WgradParams &p, int sms);

}  // namespace dg
