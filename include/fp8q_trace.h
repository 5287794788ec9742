/*
 * fp8q_trace.h -- diagnostics ABI of a TRACE build of libfp8q
 * (built with -DFP8Q_TRACE into libfp8q_trace.so; the regular library has
 * none of these symbols and no tracing code).
 *
 * Every GEMM launch of a trace build stores, for each of its first 4096
 * CTAs, 16 unsigned 64-bit slots: %globaltimer nanosecond timestamps of the
 * CTA's phases, in this order -- entry, prologue done, dependency wait
 * passed, first TMA issued, first MMA issued, last MMA committed, epilogue
 * saw the accumulator, epilogue stored/published, cluster barrier 1,
 * split-K reduction done, cluster barrier 2, exit, early weight loads
 * issued, TMEM allocated -- then, in slots 14 and 15, the SM id and the
 * CTA's rank in its cluster.  Launch i after fp8q_trace_clear() writes
 * block i % 4 of 4096 * 16 slots.  Unreached phases keep their previous
 * contents.
 *
 * Each launch also stores, for CTA 0, four slots per pipeline ring stage
 * (stages in issue order, the first 128): loads issued, MMA issuer 0 saw the
 * stage full, its commit issued, and (stages that reuse a slot) the
 * producer began waiting for the slot to be empty -- block i % 4 of 128 * 4
 * slots of a second buffer, read with fp8q_trace_read_stages.
 */
#ifndef FP8Q_TRACE_H_
#define FP8Q_TRACE_H_

#ifdef __cplusplus
extern "C" {
#endif

/* Copy `count` (<= 4 * 65536) slots of the trace buffer of the current device to
 * host memory; synchronous.  Returns 0 (FP8Q_OK) or 3 (FP8Q_ERR_CUDA). */
int fp8q_trace_read(unsigned long long *host, int count);

/* Copy `count` (<= 4 * 512) per-stage slots (see above) to host memory;
 * synchronous.  Returns 0 (FP8Q_OK) or 3 (FP8Q_ERR_CUDA). */
int fp8q_trace_read_stages(unsigned long long *host, int count);

/* Zero both trace buffers of the current device; synchronous. */
int fp8q_trace_clear(void);

#ifdef __cplusplus
}
#endif

#endif /* FP8Q_TRACE_H_ */
