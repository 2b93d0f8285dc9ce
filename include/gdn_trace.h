/* Kernel timing trace of the GatedDeltaNet layer library.
 *
 * A measurement aid; the method itself has no counterpart.  While tracing is
 * on, every kernel the library enqueues is bracketed by two CUDA events
 * recorded on the stream the kernel is launched on (the caller's stream), so
 * each kernel's device time is measured where it runs, with no added
 * synchronisation.  Events come from a pool created by gdn_trace_enable() on
 * the device that is current then; launches on another device, or beyond the
 * pool's size (GDN_TRACE_MAX_LAUNCHES), are not recorded.  Recording events is
 * not allowed inside CUDA-graph capture: leave tracing off there.
 *
 * gdn_trace_read() waits for the recorded events, adds up per kernel kind the
 * launches and their device time in milliseconds, and clears the record.
 * All functions are thread-safe (one record per process, behind a mutex).
 *
 * Returns GDN_OK, GDN_ERR_INVALID_ARG (NULL output array, cap < 1) or
 * GDN_ERR_CUDA (event creation, query or timing failed).
 */
#ifndef GDN_TRACE_H_
#define GDN_TRACE_H_

#include "gdn.h"

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  GDN_K_CHUNK_TABLE = 0, /* varlen bookkeeping: chunk table from cu_seqlens */
  GDN_K_CHUNK_PREP = 1,  /* per-chunk conv, gates, intra-chunk WY/UT terms */
  GDN_K_STATE = 2,       /* sequential inter-chunk state pass + gated RMSNorm epilogue */
  GDN_K_PREFILL_SIMT = 3,/* token-sequential fp32 prefill (inputs, the rule per column slice, the norm: 3 launches) */
  GDN_K_DECODE = 4,      /* one-token decode step */
  GDN_K_BWD_CHAIN = 5,   /* backward: inputs, forward with checkpoints, RMSNorm and the rule in reverse (4 launches) */
  GDN_K_BWD_PROLOGUE = 6,/* backward: L2 norm, SiLU and conv in reverse */
  GDN_K_SEG_SCAN = 7,    /* segment-parallel prefill: segment table and the scan over segments (2 launches) */
  GDN_K_COUNT = 8
} gdn_kernel_kind;

#define GDN_TRACE_MAX_LAUNCHES 4096

/* on != 0: create the event pool (first time) and start recording; 0: stop. */
GDN_API int gdn_trace_enable(int on);
/* launches[kind] and total_ms[kind] for kind < cap (cap >= 1, at most GDN_K_COUNT used). */
GDN_API int gdn_trace_read(int cap, int *launches, double *total_ms);
/* Name of a kernel kind ("" when out of range). */
GDN_API const char *gdn_trace_kernel_name(int kind);

#ifdef __cplusplus
}
#endif

#endif /* GDN_TRACE_H_ */
