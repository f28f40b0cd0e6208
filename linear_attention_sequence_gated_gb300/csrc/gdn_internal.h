// Internal interface between the C-ABI front end (gdn_api.cu) and the kernel
// translation units.  Not installed; not part of the ABI.
#pragma once

#include <cstddef>
#include <cstdint>
#include <mutex>
#include <cuda_runtime.h>

namespace gdn {

// Devices the library keeps per-device state for (status word, pool, kernel
// attributes); a device index at or above this is refused.
constexpr int kMaxDevices = 64;

// Index of the current device, or -1 if it cannot be read or is out of range.
inline int current_device() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return -1;
    return dev;
}

// Multiprocessors of the current device (1 if the query fails).
inline int current_sm_count() {
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
        return 1;
    return n;
}

// One-time set-up per device.  Function attributes such as the dynamic
// shared-memory opt-in apply to the device that is current when they are set,
// so each device gets its own run of `setup` (with that device current), and
// later calls on the device return the recorded result.
class PerDeviceOnce {
  public:
    template <class F>
    cudaError_t run(F &&setup) {
        const int dev = current_device();
        if (dev < 0) return cudaErrorInvalidDevice;
        std::lock_guard<std::mutex> lock(mu_);
        if (!done_[dev]) {
            err_[dev] = setup();
            done_[dev] = true;
        }
        return err_[dev];
    }

  private:
    std::mutex mu_;
    bool done_[kMaxDevices] = {};
    cudaError_t err_[kMaxDevices] = {};
};

// One validated call.  All pointers are device pointers; sizes are >= 1.
struct Problem {
    const void *q, *k;             // (B, T, Hk, d), dtype below
    const void *v;                 // (B, T, H, d), dtype below
    const float *g, *beta;         // (B, T, H)
    const float *state_in;         // (B, H, d, d) [value][key] or nullptr (zeros)
    float *out;                    // (B, T, H, d) fp32 (bf16 with out_bf16), scaled by 1/sqrt(d)
    float *state_out;              // (B, H, d, d) [value][key]; may equal state_in
    int B, T, H, Hk, d;            // value head h reads key head h % Hk (Hk divides H)
    int dtype;                     // GDN_DTYPE_F32 / GDN_DTYPE_BF16
    float scale;                   // (float)(1 / sqrt((double)d))
    int *status;                   // device status word (bounded waits report here)
    bool l2norm_qk;                // divide q and k by their norm per token first
    bool out_bf16;                 // out holds bf16: each value rounded to nearest even
};

// Recurrent path (gdn_recurrent.cu): any T >= 1, d in {32, 64, 128, 256}.
cudaError_t launch_recurrent(const Problem &p, cudaStream_t stream);

// Chunked path (gdn_chunked.cu): T >= 1, d in {64, 128, 256}.
size_t chunked_workspace_bytes(int B, int T, int H, int d, int dtype);
cudaError_t launch_chunked(const Problem &p, void *workspace, size_t ws_bytes,
                           cudaStream_t stream);
bool chunked_supports(int d);

// Value blocks of the two-kernel state walk (head_dim 256, and 128 with few
// pairs): pairs [0, pairs64) take 64-row blocks and the rest 32-row blocks,
// launched after them.
struct WalkSplit {
    int pairs64;
};
WalkSplit walk_split(long long P, int D, int sms);
// One CTA whose bounded wait gives up and records GDN_ERR_TIMEOUT (self-test).
cudaError_t launch_wait_selftest(int *status, cudaStream_t stream);

// Host-side argument checks shared by the C-ABI front ends.
namespace host {

// Bytes spanned by a dense tensor of `n` elements of `elt` bytes; false on overflow.
inline bool span_bytes(unsigned long long n, unsigned long long elt, unsigned long long *out) {
    if (n != 0 && elt > ~0ull / n) return false;
    *out = n * elt;
    return *out < (1ull << 62);
}

inline bool mul_ok(unsigned long long a, unsigned long long b, unsigned long long *out) {
    if (a != 0 && b > ~0ull / a) return false;
    *out = a * b;
    return true;
}

struct Range {
    uintptr_t lo, hi;  // [lo, hi)
};
inline bool overlap(Range a, Range b) {
    if (a.lo == a.hi || b.lo == b.hi) return false;
    return a.lo < b.hi && b.lo < a.hi;
}
inline Range range_of(const void *p, unsigned long long bytes) {
    const uintptr_t lo = reinterpret_cast<uintptr_t>(p);
    return {lo, p ? lo + (uintptr_t)bytes : lo};
}
inline bool aligned(const void *p, uintptr_t a) {
    return (reinterpret_cast<uintptr_t>(p) % a) == 0;
}

}  // namespace host

}  // namespace gdn
