/*
 * ep_signal.cuh -- device-side reads of libep's arrival signals, for a
 * consumer kernel that wants to start on destination rank d as soon as that
 * rank's rows have landed (NCCL GIN article s2.2.2 completion notification:
 * a signal is a remote-completion counter bumped by a put; s2.1.2 put with
 * SignalInc followed by waitSignal on an expected value).
 *
 * ep_signal_ptr() gives the device array signal[R]: signal[d] counts the
 * messages (TransferCmds) of every ep_dispatch since ep_create, ep_reset or
 * ep_signal_reset whose rows have landed in rank d's window.  One dispatch
 * adds sum_s msg_count[s][d] to it.  An increment is a release at GPU scope
 * made after the message's rows were written, so a thread that reads a value
 * with ep_signal_read (an acquire) sees the rows of every message it counts.
 *
 * Wait only for a dispatch that runs before the waiting kernel on its stream,
 * or inside one kernel together with the work it waits for: a kernel that
 * spins while the dispatch it waits for has not started can hold the SMs the
 * dispatch needs, and the wait then runs out.  Every wait here is bounded.
 */
#ifndef EP_SIGNAL_CUH_
#define EP_SIGNAL_CUH_

#include <stdint.h>

/* One acquire read of a signal word. */
static __device__ __forceinline__ unsigned long long ep_signal_read(const unsigned long long *signal) {
    unsigned long long v;
    asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(signal) : "memory");
    return v;
}

/* Poll *signal until it reaches `expected` or `timeout_ns` nanoseconds have
 * passed on the GPU's global timer; 100 ns back-off between reads.  Returns 1
 * if the value was reached, 0 if the wait ran out (GIN's SIGNAL_PENDING). */
static __device__ __forceinline__ int ep_signal_wait(const unsigned long long *signal, unsigned long long expected,
                                                     unsigned long long timeout_ns) {
    unsigned long long t0;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t0));
    while (true) {
        if (ep_signal_read(signal) >= expected) return 1;
        unsigned long long now;
        asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(now));
        if (now - t0 > timeout_ns) return 0;
        __nanosleep(100);
    }
}

#endif /* EP_SIGNAL_CUH_ */
