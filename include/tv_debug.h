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

/*
 * tv_debug_checks_enabled -- 1 in the index-checked build of the library
 * (compiled with -DTV_DEBUG, libtv_debug.so), 0 in the release build.
 *
 * The index-checked build tests, before each global-memory access whose
 * index a kernel computes (block-table slots, node and row indices, vocabulary
 * indices, partial-output slots, parent-pointer hops), that the index lies in
 * its array.  A failed check is counted in a device-side record of its source
 * file, the line of the first failure is kept, and the access is skipped: the
 * kernel neither traps nor faults.  In the release build every check is the
 * constant true and compiles away.
 */
int tv_debug_checks_enabled(void);

/*
 * tv_debug_check_failures -- number of failed index checks since the last
 * clear, summed over the library's source files (0 in the release build).
 * first_line / first_file (may be NULL) receive the line and the file number
 * (0 tree.cu, 1 argmax.cu, 2 attention.cu, 3 attention_tc.cu,
 * 4 attention_tc256.cu, 5 draft.cu, 6 gdn.cu; -1 none) of the first failure
 * of the first file that has one.  A non-zero `clear` zeroes the records
 * after reading them.  Synchronous: it copies the records from the current
 * device.  Returns 0xFFFFFFFF when a copy fails.
 */
unsigned tv_debug_check_failures(unsigned *first_line, int *first_file, int clear);

#ifdef __cplusplus
}
#endif

#endif /* TV_DEBUG_H_ */
