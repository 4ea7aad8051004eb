// attn_sync.cuh -- bounded mbarrier waits shared by the attention kernels.
//
// Every wait of a kernel role is bounded. The first kSpinProbes probes are plain try_waits (the
// hardware holds the thread briefly and wakes it as the phase completes: the lowest latency for
// the short waits of the steady state); later probes park the thread for up to kProbeNs each.
// Every probe counts toward the plan's wait limit; reaching it expires the wait: the CTA records
// an error (sticky status word, first writer wins), raises its abort flag and the launch-wide
// abort word, and every role unwinds. A limit shorter than the spin phase (a test configuration)
// makes every probe a non-blocking poll, so that the limit counts polls exactly.
#pragma once

#include "sm103_ptx.cuh"

namespace falp {
namespace {

constexpr uint32_t kProbeNs = 100000;     // one parked probe: at most ~100 us
constexpr int kSpinProbes = 64;           // plain probes before parking
constexpr long long kDrainProbes = 20000; // drains give up after ~2 s

struct WaitCtx {
  int* err;          // sticky error word of the plan (read and cleared by the host)
  int* abort_word;   // launch generation that aborted, shared by every CTA of the launch
  int gen;           // this launch's generation
  long long spin_limit;
};

// Out-of-line part of wait_phase (keeps the inlined fast path small).
__device__ __noinline__ bool wait_phase_slow(uint32_t bar, uint32_t parity, int* abort_flag,
                                             const WaitCtx& a, int role) {
  const bool exact = a.spin_limit < kSpinProbes;
  long long n = exact ? 0 : 1;  // the inlined fast path made one probe already
  for (;;) {
    if (n >= a.spin_limit) {
      *reinterpret_cast<volatile int*>(abort_flag) = 1;
      atomicExch(a.abort_word, a.gen);
      atomicCAS(a.err, 0, 0x100 | role);
      return false;
    }
    const bool parked = n >= kSpinProbes;
    bool done;
    if (exact) done = mbar_test_wait(bar, parity);
    else if (parked) done = mbar_try_wait_sleep(bar, parity, kProbeNs);
    else done = mbar_try_wait(bar, parity);
    if (done) return true;
    ++n;
    if (parked) {
      if (*reinterpret_cast<volatile int*>(abort_flag)) return false;
      if (*reinterpret_cast<volatile int*>(a.abort_word) == a.gen) {  // another CTA gave up
        *reinterpret_cast<volatile int*>(abort_flag) = 1;
        return false;
      }
    }
  }
}

// Bounded wait on one mbarrier phase; false when the CTA aborts (this wait expired, or another
// wait of this launch did).
__device__ __forceinline__ bool wait_phase(uint32_t bar, uint32_t parity, int* abort_flag,
                                           const WaitCtx& a, int role) {
  if (a.spin_limit >= kSpinProbes && mbar_try_wait(bar, parity)) return true;
  return wait_phase_slow(bar, parity, abort_flag, a, role);
}

// Wait used while draining after an abort: ignores the abort flag, bounded separately.
__device__ __forceinline__ void drain_phase(uint32_t bar, uint32_t parity) {
  for (long long n = 0; n < kDrainProbes; ++n)
    if (mbar_try_wait_sleep(bar, parity, kProbeNs)) return;
}

}  // namespace
}  // namespace falp
