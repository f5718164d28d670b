// Test helper, not part of the library: one warp that lets the next kernel on
// the stream start at once (programmatic dependent launch) and then keeps its
// own grid alive for a set time, read from the global timer.  The dependent
// kernel's CTAs run meanwhile, but whatever they order behind
// griddepcontrol.wait (the library's kernels: their first reads of data an
// earlier kernel may write) waits until this kernel ends.  A consumer wait of
// the dependent kernel that lies behind such a read therefore lasts the whole
// hold -- a wait that genuinely runs past a short limit, with nothing faulted.
// The hold ends by itself: its only loop is bounded by the timer.
#include <cuda_runtime.h>
#include <stdint.h>

__global__ void pdl_hold_kernel(unsigned long long ns) {
  asm volatile("griddepcontrol.launch_dependents;");
  uint64_t t0, t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t0));
  do {
    __nanosleep(1000);
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  } while (t - t0 < ns);
}

extern "C" int pdl_hold(unsigned long long ns, void* stream) {
  if (ns > 1000000000ull) return (int)cudaErrorInvalidValue;   // at most a second
  pdl_hold_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(ns);
  return (int)cudaGetLastError();
}
