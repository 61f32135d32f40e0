// Internal layout structures shared by the host planner (plan.cpp) and the
// device side (kernels.cu).  Not part of the C ABI.
#pragma once

#include <atomic>
#include <cstdint>
#include <string>
#include <vector>

#include "fsdp_pack.h"

namespace fsdp {

// Element-type pair of one work item: bit 0 = source is BF16, bit 1 =
// destination is BF16.
enum Kind : uint8_t {
  KIND_F32_F32 = 0,
  KIND_BF16_F32 = 1,
  KIND_F32_BF16 = 2,
  KIND_BF16_BF16 = 3,
};

inline uint8_t kind_of(int32_t src_dtype, int32_t dst_dtype) {
  return (uint8_t)((src_dtype == FSDP_DTYPE_BF16 ? 1 : 0) | (dst_dtype == FSDP_DTYPE_BF16 ? 2 : 0));
}

inline int64_t dtype_bytes(int32_t dt) { return dt == FSDP_DTYPE_F32 ? 4 : 2; }

// One contiguous run of a copy: dst[k] = k < n_copy ? cast(src[k]) : 0 for
// k < n_total, where src and dst are the slot pointers advanced by the
// element offsets.  Source and destination pointers travel per call in the
// kernel's parameter block; items name them by slot.
struct alignas(16) WorkItem {
  int64_t src_off;    // elements into the source slot
  int64_t dst_off;    // elements into the destination slot
  int32_t n_copy;     // leading destination elements that come from the source
  int32_t n_total;    // destination elements written (the rest are +0)
  uint16_t src_slot;
  uint16_t dst_slot;
  uint8_t kind;
  uint8_t reserved[3];
};
static_assert(sizeof(WorkItem) == 32, "work item must stay 32 bytes");

// Size limits of one work item.  Its source bytes are staged whole in one
// shared-memory stage of the kernel's pipeline, so they may not exceed
// kStageBytes; its destination bytes are bounded too so that long runs split
// into pieces that balance across the grid.
constexpr int64_t kStageBytes = 16 * 1024;
constexpr int64_t kItemDstBytes = 16 * 1024;

enum Op { OP_PACK = 0, OP_COPY_IN = 1, OP_COPY_OUT = 2, OP_RS_COPY_OUT = 3, OP_COUNT = 4 };

struct OpTable {
  int64_t first = 0;   // index of the op's first item in the shared table
  int64_t count = 0;   // items of the op
  int32_t n_slots = 0; // pointer slots the op's launch carries
  int32_t grid = 0;    // CTAs per launch
};

struct ParamPlan {
  int64_t chunk = 0;
  int32_t bucket = 0;
  int32_t group = 0;
  int64_t bucket_off = 0;
  int64_t group_off = 0;
};

struct BucketPlan {
  int32_t dtype = 0;
  int32_t n_params = 0;
  int64_t S = 0;
};

struct GroupPlan {
  int32_t shard_dtype = 0;
  int32_t param_dtype = 0;
  int32_t n_params = 0;
  int64_t byte_off = 0;
  int64_t elems = 0;
};

}  // namespace fsdp

struct fsdp_layout {
  int32_t W = 1;
  int32_t device = -1;           // -1: host-only layout
  std::vector<fsdp_param_desc_t> desc;
  std::vector<fsdp::ParamPlan> param;
  std::vector<fsdp::BucketPlan> bucket;
  std::vector<fsdp::GroupPlan> group;
  int64_t S_ag = 0;
  std::vector<fsdp::WorkItem> items;   // pack, copy-in, copy-out, rs copy-out tables back to back
  fsdp::OpTable op[fsdp::OP_COUNT];
  int64_t resident = 0;                // CTAs a launch keeps resident on the device
  int32_t sms = 0;                     // SMs of the device
  fsdp::WorkItem *d_items = nullptr;   // device copy of `items`
  uint32_t *d_status = nullptr;        // device status word (bounded-wait failures)
  unsigned long long *d_sched = nullptr;  // one work-sharing word per operation (device)
  // Host counters of the owner tags that launches put in those words.
  mutable std::atomic<uint32_t> sched_epoch[fsdp::OP_COUNT]{};
};

namespace fsdp {
// Thread-local error reporting used by every entry point.
fsdp_status_t fail(fsdp_status_t st, const std::string &msg);
void clear_error();

// Device side (kernels.cu): choose grids and upload the work table.
fsdp_status_t device_setup(fsdp_layout *L);
void device_release(fsdp_layout *L);

// Host-side argument checks of the entry points (kernels.cu): the layout has
// a device table on the current device; p is non-NULL (when bytes > 0) and
// aligned to `align` bytes.  `what` and `index` name the argument in the
// error message (index < 0: no index).
fsdp_status_t check_layout(const fsdp_layout *L);
fsdp_status_t check_ptr(const void *p, int64_t bytes, int64_t align, const char *what, int64_t index);
}  // namespace fsdp
