/*
 * fp8pa_testing — test, tuning and profiling hooks of libfp8pa.
 *
 * These calls are not part of the product interface in fp8pa.h.  They exist
 * so that the library's own tests and benchmark can time kernels, force a
 * kernel variant or exercise the bounded-wait timeout path.  Every hook
 * changes only the later calls made FROM THE CALLING HOST THREAD: another
 * thread's calls (and the kernels a CUDA graph captured earlier) are not
 * affected.  Each setting stays in force on that thread until it is set
 * again; 0 (or NULL) restores the default.
 *
 * None of these has a counterpart on the source pages.
 */
#ifndef FP8PA_TESTING_H_
#define FP8PA_TESTING_H_

#ifdef __cplusplus
extern "C" {
#endif

/*
 * fp8pa_set_timing_events — profiling hook.  When both are non-NULL
 * (cudaEvent_t handles), later fp8_paged_attn_fwd calls on this thread record
 * `start` on their stream just before the first attention kernel and `stop`
 * just after the last one, so the caller can time the attention kernels
 * alone.  NULL, NULL turns it off.
 */
void fp8pa_set_timing_events(void* start_event, void* stop_event);

/*
 * fp8pa_set_ctas_per_sm — tuning hook: 1 or 2 forces that many attention CTAs
 * per SM where the kernel variant supports it; 0 restores the automatic choice
 * (two co-resident CTAs for E4M3 Q with 16-row tiles, else one).  Results do
 * not depend on it.
 */
void fp8pa_set_ctas_per_sm(int ctas);

/*
 * fp8pa_set_bf16_dequant_v — selects the form of the BF16-Q path.  0 (default):
 * Q is split per row into an exact E4M3 pair and QK^T runs as FP8 MMAs on the
 * E4M3 K; V stays E4M3, exact, in an E4M3 PV MMA with P carried as an E4M3
 * hi/lo pair (about BF16's 8 significant bits).  1: the literal dequant form,
 * kept to check the default against: Q in F16, K dequantized to F16 in tensor
 * memory for a 16-bit QK^T, V dequantized to BF16 in shared memory and PV a BF16
 * MMA with BF16 P.
 */
void fp8pa_set_bf16_dequant_v(int on);

/*
 * fp8pa_set_grid_sms — tuning hook: the attention kernels' persistent grids use
 * at most this many SMs (0 = all).  Results do not depend on it; it measures
 * how a workload's throughput scales with the SMs it gets.
 */
void fp8pa_set_grid_sms(int sms);

/*
 * fp8pa_set_prefill_rows — tuning hook: packed query rows per tile of
 * prefill-class row tiles with BF16 Q, 32 or 64 (0 = the default, 64).  Results
 * agree within rounding; it measures the tile size's cost.
 */
void fp8pa_set_prefill_rows(int rows);

/*
 * fp8pa_set_sm_split — tuning hook: when a call runs its decode and prefill row
 * classes side by side, the prefill class gets this many SMs instead of the
 * plan kernel's estimate (0 = the estimate).  Results do not depend on it.
 */
void fp8pa_set_sm_split(int sms);

/*
 * fp8pa_set_wait_limit — test hook.  Sets the iteration cap of every bounded
 * pipeline wait in later launches (0 restores the default).  A tiny cap makes
 * waits run out, which exercises the timeout path: the kernel sets
 * FP8PA_DEV_TIMEOUT, drains its own copies and MMAs, frees its tensor memory
 * and returns; results of that launch are undefined.
 */
void fp8pa_set_wait_limit(unsigned int max_iterations);

/*
 * fp8pa_set_stall_injection — test hook (0 = off, the default).  While on, the
 * MMA-issuing thread of every attention CTA of later launches first waits on a
 * barrier that nothing ever arrives on, so that wait always runs out (after the
 * wait limit above or about two seconds, whichever comes first).  The launch
 * then takes the timeout path described above: FP8PA_DEV_TIMEOUT is set, the
 * call itself returns OK, results of that launch are undefined, and the CUDA
 * context stays usable.
 */
void fp8pa_set_stall_injection(int on);

#ifdef __cplusplus
}
#endif

#endif /* FP8PA_TESTING_H_ */
