// Host-side glue shared by the forward, backward and API translation units.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>

#include "../../include/fa.h"

namespace fa {

constexpr int kTile = 128;  // rows of a query tile and of a key/value tile

// Failure-path test hooks.  Only a separate test build of the library
// (compiled with FA_TEST_HOOKS) can make a producer withhold one load, so that
// a barrier is never completed and the kernel's bounded waits must expire;
// the product build has neither the switch nor the code behind it.
enum TestWithhold : int { kWithholdNone = 0, kWithholdFwdQ = 1, kWithholdBwdDO = 2 };
#ifdef FA_TEST_HOOKS
int test_withhold();
#else
constexpr int test_withhold() { return kWithholdNone; }
#endif

struct Problem {
  int B, Hq, Hkv, Tq, Tk, d, dv;  // d: Q/K head size, dv: V/O head size
  int causal;
  int window;   // causal sliding window in keys, 0 = none
  float scale;  // resolved (> 0)
  int G() const { return Hq / Hkv; }
  int q_tiles() const { return (Tq + kTile - 1) / kTile; }
  int kv_tiles() const { return (Tk + kTile - 1) / kTile; }
  long long Tq_pad() const { return (long long)q_tiles() * kTile; }
};

// Encodes a TMA descriptor for a contiguous bf16 tensor viewed as
// [outer][rows][inner] (inner contiguous), box = 64 x 128 x 1, 128-byte swizzle.
// Returns false if cuTensorMapEncodeTiled rejects it.
bool encode_rows_bf16(CUtensorMap* map, const void* base, int inner, int rows, long long outer);

// TMA descriptor for the fp32 dQ accumulator viewed as [outer][rows][inner]
// (inner = d), box = 32 x box_rows x 1 (128 bytes x box_rows), 128-byte swizzle.
bool encode_acc_f32(CUtensorMap* map, const void* base, int inner, long long rows, long long outer, int box_rows);

// Device status word of the current device (see fa_last_device_status).
int* device_status_word();

// Lets `kernel` use `bytes` of dynamic shared memory on the current device.
// The attribute is per device, so it is set once for each (kernel, device)
// pair; safe to call from several host threads.
cudaError_t allow_dynamic_smem(const void* kernel, int bytes);

// Launchers.  Each returns the first CUDA error it met and adds the number
// of kernels it enqueued to *launches.
cudaError_t launch_forward(const Problem& p, const void* Q, const void* K, const void* V, void* O, float* L,
                           cudaStream_t stream, int* launches);
// `workspace_bytes` decides whether the split-item area fits (see BwdWorkspace).
cudaError_t launch_backward(const Problem& p, const void* Q, const void* K, const void* V, const void* O,
                            const void* dO, const float* L, void* dQ, void* dK, void* dV, void* workspace,
                            size_t workspace_bytes, int stages, cudaStream_t stream, int* launches);

// Groups per super-batch of the backward's grid order: the smallest divisor
// S of n_groups with S * kv_tiles >= 1.5 * sms, searched up to four times the
// least such S; n_groups (a single super-batch) when there is none.
inline int super_batch_groups(int n_groups, int kv_tiles, int sms) {
  if (n_groups < 1 || kv_tiles < 1) return n_groups;
  const long long want = (3LL * sms + 1) / 2;
  const long long s_min = want <= kv_tiles ? 1 : (want + kv_tiles - 1) / kv_tiles;
  for (long long s = s_min; s < n_groups && s <= 4 * s_min; ++s)
    if (n_groups % s == 0) return (int)s;
  return n_groups;
}

// Work items of the backward main kernel that may be split in two (see
// backward_split_items); the workspace holds their fp32 partial dK / dV.
constexpr int kMaxSplitItems = 128;

// Workspace carve-up of fa_backward (byte offsets, 256-aligned).  `part` and
// `counters` (the split items' partial dK / dV and their finish counters)
// are empty when no item can be split (with a causal mask).  The backward
// needs `total_min` bytes (up to `part`); it splits items only when the
// workspace also holds the split area (`total`).
struct BwdWorkspace {
  size_t dq_acc, lse2, delta, part, counters, total_min, total;
  int split_cap;  // items the partial area has room for
};
BwdWorkspace backward_workspace_layout(const Problem& p);

}  // namespace fa
