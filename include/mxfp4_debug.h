/*
 * mxfp4_debug.h — extra entry point of the bounds-checking build of the
 * library (libmxfp4_gb300_debug.so, compiled with -DMXFP4_DEBUG_BOUNDS).
 *
 * That build exports everything in mxfp4.h with identical results, and in
 * addition checks every global-memory access of every kernel against the
 * byte range its buffer has according to the call's arguments (the ranges
 * the host-side validation also uses).  An access outside its range is not
 * performed (a load reads zeros) and is counted; no kernel traps.  It is a
 * testing aid in place of an external memory checker, and slower
 * than the normal build.  No counterpart exists in the method's sources.
 */
#ifndef MXFP4_GB300_DEBUG_H
#define MXFP4_GB300_DEBUG_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Synchronises the current device, then returns the number of out-of-range
 * accesses every kernel of the library attempted since the previous call
 * (and resets the count), or -1 when the synchronisation reports an error. */
int64_t mxfp4_debug_bounds_violations(void);

#ifdef __cplusplus
}
#endif

#endif /* MXFP4_GB300_DEBUG_H */
