/*
 * smq_trace.h: phase timestamps of the gather + score kernel, exported only
 * by the tracing build of the library (libsmq_trace.so, compiled with
 * -DSMQ_TRACE by sparse_attention_top_expand_gb300/csrc/build.py
 * build(trace=True)). The product library exports neither call.
 *
 * In the tracing build each CTA of the score kernel writes %globaltimer
 * (nanoseconds) into its own row of 32 slots of a device array when it
 * passes a phase boundary; a later launch overwrites the rows of its CTAs.
 * Slots (0 = never stamped):
 *   0 entry            1 after the grid-dependency wait   2 tile range known
 *   3 TMEM and query-scale set-up done   4 scheduler: first row expanded
 *   5 scheduler: first tile published    6 scheduler: last tile published
 *   7 loaders: first stage filled        8 loaders: last stage filled
 *   9 MMA: first tile committed         10 MMA: last tile committed
 *  11 epilogue: first tile stored       12 epilogue: last tile stored
 *  13 pipeline torn down                14 top-k: a row's selection starts
 *  15 top-k: a row's selection ends     16 exit
 */
#ifndef SMQ_TRACE_H
#define SMQ_TRACE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#ifdef SMQ_TRACE
/* Copy the first `count` stamps (CTA-major, 32 per CTA, at most 1024 CTAs)
 * to host memory. Synchronous. */
__attribute__((visibility("default"))) int smq_trace_read(uint64_t *host, size_t count);
/* Zero every stamp. Synchronous. */
__attribute__((visibility("default"))) int smq_trace_clear(void);
#endif

#ifdef __cplusplus
}
#endif

#endif /* SMQ_TRACE_H */
