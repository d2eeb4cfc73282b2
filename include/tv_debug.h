/*
 * tv_debug.h -- test hooks of libtv.  Nothing in a verify step calls them;
 * they exist so that tests can drive code paths that correct inputs never
 * reach, without faulting or hanging a GPU.
 */
#ifndef TV_DEBUG_H_
#define TV_DEBUG_H_

#ifdef __cplusplus
extern "C" {
#endif

/*
 * tv_debug_withhold_arrival -- exercise the bounded-wait expiry path of the
 * tensor-core kernels (the D = 128 and D = 256 tree-attention kernels and the
 * pipelined GDN tree-verify kernel).
 *
 * From the next launch on, in the CTA with linear index `cta` (blockIdx.x +
 * blockIdx.y * gridDim.x) the mbarrier that signals the first K/V copy
 * (attention) or the first state copy (GDN) is initialised to expect one
 * arrival more than the producer makes.  The copy still lands, but the phase
 * never completes: the consumer's wait runs out after its bound (2 s), the
 * CTA raises its abort flag, every role leaves its loop, copies in flight get
 * a bounded chance to land, issued MMAs are waited for, the tensor memory is
 * freed, and TV_ERR_CUDA is recorded in status[] of the sequence being worked
 * on.  Other CTAs run normally.  A negative `cta` (the initial state)
 * disarms it.  Host-side state of the process, read at every launch; not
 * thread-safe with respect to launches running concurrently in other threads.
 * The pages have no counterpart to this call: it tests this library.
 */
void tv_debug_withhold_arrival(int cta);

#ifdef __cplusplus
}
#endif

#endif /* TV_DEBUG_H_ */
