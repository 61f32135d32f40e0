// Host planner: per-parameter chunks, reduce-scatter buckets, all-gather
// dtype groups, and the work tables that the kernels walk.
//
// Layout rules ("The unit you wrapped", FlatParameter and padding sections;
// "FSDP2 per-parameter mixed precision" news item, paragraphs 1-2):
//   c_p = ceil(n_p / W); rank r owns flat elements [r*c_p, (r+1)*c_p) of the
//   parameter padded on the right to W*c_p.
//   One bucket per distinct reduce dtype (first appearance), parameters in
//   registration order inside it.
//   One all-gather group per distinct (shard dtype, param dtype) pair (first
//   appearance); groups start on 16-byte boundaries inside a rank's row.
#include <algorithm>
#include <cstring>
#include <new>

#include "layout.h"

namespace fsdp {

namespace {

thread_local std::string g_last_error;

int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }
int64_t align_up(int64_t x, int64_t a) { return ceil_div(x, a) * a; }

bool valid_dtype(int32_t dt) { return dt == FSDP_DTYPE_F32 || dt == FSDP_DTYPE_BF16; }

// Split the run [0, n_total) of destination elements into work items of at
// most kItemDstBytes of destination and kStageBytes of source.  Interior cut
// points fall on 256-byte boundaries of the destination (relative to the slot
// base) so that only the first piece of a run can start unaligned.
void emit_run(std::vector<WorkItem> &out, int64_t src_off, int64_t dst_off, int64_t n_copy,
              int64_t n_total, uint16_t src_slot, uint16_t dst_slot, uint8_t kind,
              int64_t dst_elem_bytes) {
  const int64_t src_elem_bytes = (kind & 1) ? 2 : 4;
  const int64_t max_elems = std::min(kItemDstBytes / dst_elem_bytes, kStageBytes / src_elem_bytes);
  const int64_t align = 256 / dst_elem_bytes;
  int64_t start = 0;
  while (start < n_total) {
    const int64_t remaining = n_total - start;
    int64_t end = n_total;
    if (remaining > max_elems) {
      // Even split of what is left, cut down to an aligned destination
      // element; never longer than max_elems.
      const int64_t pieces_left = ceil_div(remaining, max_elems);
      end = (dst_off + start + ceil_div(remaining, pieces_left)) / align * align - dst_off;
      if (end <= start) end = start + max_elems;
      end = std::min(end, start + max_elems);
    }
    WorkItem w{};
    w.src_off = src_off + start;
    w.dst_off = dst_off + start;
    w.n_total = (int32_t)(end - start);
    w.n_copy = (int32_t)std::max<int64_t>(0, std::min(n_copy, end) - start);
    w.src_slot = src_slot;
    w.dst_slot = dst_slot;
    w.kind = kind;
    out.push_back(w);
    start = end;
  }
}

// Self-check of the work tables: for every output (bucket buffer, all-gather
// row, full parameter) the items that write it must tile its bytes exactly
// once, and no item may stage more source bytes than one pipeline stage.
bool tables_consistent(const fsdp_layout &L) {
  struct Span {
    int64_t begin, end;
  };
  const int32_t P = (int32_t)L.desc.size(), B = (int32_t)L.bucket.size();
  for (int op = 0; op < OP_COUNT; ++op) {
    // Output slots of this op and their sizes in bytes.
    std::vector<int64_t> out_bytes;
    int32_t first_out = 0;
    if (op == OP_PACK) {
      first_out = P;
      for (int32_t b = 0; b < B; ++b) out_bytes.push_back((int64_t)L.W * L.bucket[b].S * dtype_bytes(L.bucket[b].dtype));
    } else if (op == OP_COPY_IN) {
      first_out = P;
      out_bytes.push_back(L.S_ag);
    } else if (op == OP_COPY_OUT) {
      first_out = 1;
      for (int32_t p = 0; p < P; ++p) out_bytes.push_back(L.desc[p].numel * dtype_bytes(L.desc[p].param_dtype));
    } else {
      first_out = B;
      for (int32_t p = 0; p < P; ++p) out_bytes.push_back(L.param[p].chunk * dtype_bytes(L.desc[p].shard_dtype));
    }
    std::vector<std::vector<Span>> spans(out_bytes.size());
    for (int64_t i = L.op[op].first; i < L.op[op].first + L.op[op].count; ++i) {
      const WorkItem &w = L.items[i];
      const int64_t ss = (w.kind & 1) ? 2 : 4, ds = (w.kind & 2) ? 2 : 4;
      if (w.n_total <= 0 || w.n_copy < 0 || w.n_copy > w.n_total) return false;
      if ((int64_t)w.n_copy * ss > kStageBytes || (int64_t)w.n_total * ds > kItemDstBytes) return false;
      const int64_t o = (int64_t)w.dst_slot - first_out;
      if (o < 0 || o >= (int64_t)out_bytes.size()) return false;
      spans[o].push_back({w.dst_off * ds, (w.dst_off + w.n_total) * ds});
    }
    for (size_t o = 0; o < spans.size(); ++o) {
      std::sort(spans[o].begin(), spans[o].end(), [](const Span &x, const Span &y) { return x.begin < y.begin; });
      int64_t at = 0;
      for (const Span &sp : spans[o]) {
        if (sp.begin != at) return false;
        at = sp.end;
      }
      if (at != out_bytes[o]) return false;
    }
  }
  return true;
}

fsdp_status_t plan(const fsdp_param_desc_t *params, const int64_t *row_elems, int32_t n, int32_t W,
                   bool with_device, fsdp_layout_t **out) {
  if (!out) return fail(FSDP_EINVAL, "out is NULL");
  *out = nullptr;
  if (n < 0) return fail(FSDP_EINVAL, "n_params < 0");
  if (n > FSDP_MAX_PARAMS) return fail(FSDP_EUNSUPPORTED, "n_params > FSDP_MAX_PARAMS");
  if (W < 1) return fail(FSDP_EINVAL, "world_size < 1");
  if (n > 0 && !params) return fail(FSDP_EINVAL, "params is NULL");
  for (int32_t p = 0; p < n; ++p) {
    const fsdp_param_desc_t &d = params[p];
    if (d.numel < 0) return fail(FSDP_EINVAL, "params[" + std::to_string(p) + "].numel < 0");
    if (!valid_dtype(d.grad_dtype) || !valid_dtype(d.reduce_dtype) || !valid_dtype(d.shard_dtype) ||
        !valid_dtype(d.param_dtype))
      return fail(FSDP_EINVAL, "params[" + std::to_string(p) + "] has an unknown dtype");
    // Each item carries 32-bit element counts of one rank's run; a chunk is
    // split into items, so only the byte offsets below need 64 bits.
    if (d.numel > (int64_t(1) << 46))
      return fail(FSDP_EUNSUPPORTED, "params[" + std::to_string(p) + "].numel above 2^46");
    if (row_elems && (row_elems[p] < 0 || (row_elems[p] > 0 && d.numel % row_elems[p] != 0)))
      return fail(FSDP_EINVAL, "row_elems[" + std::to_string(p) + "] is negative or does not divide numel");
  }

  fsdp_layout *L = new (std::nothrow) fsdp_layout();
  if (!L) return fail(FSDP_ENOMEM, "host allocation failed");
  try {
    L->W = W;
    L->desc.assign(params, params + n);
    L->param.resize(n);
    // Chunks, buckets and groups, in registration order.
    for (int32_t p = 0; p < n; ++p) {
      const fsdp_param_desc_t &d = params[p];
      ParamPlan &pp = L->param[p];
      // Flattened: ceil(n_p / W) elements.  Row chunks: ceil(d0 / W) rows of
      // row_elems elements, d0 = n_p / row_elems.
      if (row_elems && row_elems[p] > 0)
        pp.chunk = ceil_div(d.numel / row_elems[p], W) * row_elems[p];
      else
        pp.chunk = ceil_div(d.numel, W);
      int32_t b = -1;
      for (size_t k = 0; k < L->bucket.size(); ++k)
        if (L->bucket[k].dtype == d.reduce_dtype) b = (int32_t)k;
      if (b < 0) {
        b = (int32_t)L->bucket.size();
        BucketPlan nb;
        nb.dtype = d.reduce_dtype;
        L->bucket.push_back(nb);
      }
      pp.bucket = b;
      pp.bucket_off = L->bucket[b].S;
      L->bucket[b].S += pp.chunk;
      L->bucket[b].n_params += 1;
      int32_t g = -1;
      for (size_t k = 0; k < L->group.size(); ++k)
        if (L->group[k].shard_dtype == d.shard_dtype && L->group[k].param_dtype == d.param_dtype)
          g = (int32_t)k;
      if (g < 0) {
        g = (int32_t)L->group.size();
        GroupPlan ng;
        ng.shard_dtype = d.shard_dtype;
        ng.param_dtype = d.param_dtype;
        L->group.push_back(ng);
      }
      pp.group = g;
      pp.group_off = L->group[g].elems;
      L->group[g].elems += pp.chunk;
      L->group[g].n_params += 1;
    }
    int64_t end = 0;
    for (GroupPlan &g : L->group) {
      g.byte_off = align_up(end, 16);
      end = g.byte_off + g.elems * dtype_bytes(g.param_dtype);
    }
    L->S_ag = align_up(end, 16);

    // Work tables.  Slots: pack = [grads 0..P) [buckets P..P+B);
    // copy-in = [shards 0..P) [ag_input P]; copy-out = [ag_output 0] [params 1..P].
    std::vector<WorkItem> &items = L->items;
    const int32_t P = n, B = (int32_t)L->bucket.size();

    L->op[OP_PACK].first = (int64_t)items.size();
    for (int32_t b = 0; b < B; ++b)
      for (int32_t r = 0; r < W; ++r)
        for (int32_t p = 0; p < P; ++p) {
          const ParamPlan &pp = L->param[p];
          if (pp.bucket != b || pp.chunk == 0) continue;
          int64_t first = (int64_t)r * pp.chunk;
          int64_t n_copy = std::max<int64_t>(0, std::min(pp.chunk, params[p].numel - first));
          emit_run(items, first, (int64_t)r * L->bucket[b].S + pp.bucket_off, n_copy, pp.chunk,
                   (uint16_t)p, (uint16_t)(P + b), kind_of(params[p].grad_dtype, L->bucket[b].dtype),
                   dtype_bytes(L->bucket[b].dtype));
        }
    L->op[OP_PACK].count = (int64_t)items.size() - L->op[OP_PACK].first;
    L->op[OP_PACK].n_slots = P + B;

    L->op[OP_COPY_IN].first = (int64_t)items.size();
    int64_t cursor = 0;  // bytes of the row written so far
    for (size_t g = 0; g < L->group.size(); ++g) {
      const GroupPlan &gp = L->group[g];
      // Zero the alignment gap before the group (an even number of bytes).
      if (gp.byte_off > cursor)
        emit_run(items, 0, cursor / 2, 0, (gp.byte_off - cursor) / 2, 0, (uint16_t)P, KIND_BF16_BF16, 2);
      const int64_t sz = dtype_bytes(gp.param_dtype);
      for (int32_t p = 0; p < P; ++p) {
        const ParamPlan &pp = L->param[p];
        if (pp.group != (int32_t)g) continue;
        emit_run(items, 0, gp.byte_off / sz + pp.group_off, pp.chunk, pp.chunk, (uint16_t)p,
                 (uint16_t)P, kind_of(gp.shard_dtype, gp.param_dtype), sz);
      }
      cursor = gp.byte_off + gp.elems * sz;
    }
    if (L->S_ag > cursor)
      emit_run(items, 0, cursor / 2, 0, (L->S_ag - cursor) / 2, 0, (uint16_t)P, KIND_BF16_BF16, 2);
    L->op[OP_COPY_IN].count = (int64_t)items.size() - L->op[OP_COPY_IN].first;
    L->op[OP_COPY_IN].n_slots = P + 1;

    L->op[OP_COPY_OUT].first = (int64_t)items.size();
    for (int32_t p = 0; p < P; ++p) {
      const ParamPlan &pp = L->param[p];
      const GroupPlan &gp = L->group[pp.group];
      const int64_t sz = dtype_bytes(gp.param_dtype);
      for (int32_t r = 0; r < W; ++r) {
        int64_t first = (int64_t)r * pp.chunk;
        int64_t valid = std::max<int64_t>(0, std::min(pp.chunk, params[p].numel - first));
        emit_run(items, ((int64_t)r * L->S_ag + gp.byte_off) / sz + pp.group_off, first, valid, valid,
                 0, (uint16_t)(1 + p), kind_of(gp.param_dtype, gp.param_dtype), sz);
      }
    }
    L->op[OP_COPY_OUT].count = (int64_t)items.size() - L->op[OP_COPY_OUT].first;
    L->op[OP_COPY_OUT].n_slots = P + 1;

    // Reduce-scatter copy-out: slots [reduced rows 0..B) [sharded grads B..B+P).
    L->op[OP_RS_COPY_OUT].first = (int64_t)items.size();
    for (int32_t p = 0; p < P; ++p) {
      const ParamPlan &pp = L->param[p];
      emit_run(items, pp.bucket_off, 0, pp.chunk, pp.chunk, (uint16_t)pp.bucket, (uint16_t)(B + p),
               kind_of(L->bucket[pp.bucket].dtype, params[p].shard_dtype), dtype_bytes(params[p].shard_dtype));
    }
    L->op[OP_RS_COPY_OUT].count = (int64_t)items.size() - L->op[OP_RS_COPY_OUT].first;
    L->op[OP_RS_COPY_OUT].n_slots = B + P;
  } catch (const std::bad_alloc &) {
    delete L;
    return fail(FSDP_ENOMEM, "host allocation failed while planning");
  }
  if (!tables_consistent(*L)) {
    delete L;
    return fail(FSDP_EUNSUPPORTED, "internal error: work tables do not tile the outputs");
  }

  if (with_device) {
    fsdp_status_t st = device_setup(L);
    if (st != FSDP_OK) {
      delete L;
      return st;
    }
  }
  *out = L;
  clear_error();
  return FSDP_OK;
}

}  // namespace

fsdp_status_t fail(fsdp_status_t st, const std::string &msg) {
  g_last_error = msg;
  return st;
}

void clear_error() { g_last_error.clear(); }

}  // namespace fsdp

using namespace fsdp;

extern "C" {

fsdp_status_t fsdp_plan_layout(const fsdp_param_desc_t *params, int32_t n_params, int32_t world_size,
                               fsdp_layout_t **out) {
  return plan(params, nullptr, n_params, world_size, true, out);
}

fsdp_status_t fsdp_plan_layout_host(const fsdp_param_desc_t *params, int32_t n_params,
                                    int32_t world_size, fsdp_layout_t **out) {
  return plan(params, nullptr, n_params, world_size, false, out);
}

fsdp_status_t fsdp_plan_layout_ex(const fsdp_param_desc_t *params, const int64_t *row_elems, int32_t n_params,
                                  int32_t world_size, uint32_t flags, fsdp_layout_t **out) {
  if (flags & ~(uint32_t)FSDP_PLAN_HOST_ONLY) return fail(FSDP_EINVAL, "unknown plan flags");
  return plan(params, row_elems, n_params, world_size, (flags & FSDP_PLAN_HOST_ONLY) == 0, out);
}

fsdp_status_t fsdp_layout_query(const fsdp_layout_t *L, fsdp_layout_info_t *info) {
  if (!L || !info) return fail(FSDP_EINVAL, "NULL layout or info");
  std::memset(info, 0, sizeof(*info));
  info->world_size = L->W;
  info->n_params = (int32_t)L->desc.size();
  info->n_buckets = (int32_t)L->bucket.size();
  info->n_groups = (int32_t)L->group.size();
  info->ag_bytes = L->S_ag;
  for (const fsdp_param_desc_t &d : L->desc) info->total_numel += d.numel;
  info->device = L->device;
  info->has_device_table = (L->device >= 0) ? 1 : 0;
  info->pack_items = L->op[OP_PACK].count;
  info->copy_in_items = L->op[OP_COPY_IN].count;
  info->copy_out_items = L->op[OP_COPY_OUT].count;
  info->rs_copy_out_items = L->op[OP_RS_COPY_OUT].count;
  clear_error();
  return FSDP_OK;
}

fsdp_status_t fsdp_layout_param(const fsdp_layout_t *L, int32_t p, fsdp_param_info_t *info) {
  if (!L || !info) return fail(FSDP_EINVAL, "NULL layout or info");
  if (p < 0 || p >= (int32_t)L->param.size()) return fail(FSDP_EINVAL, "parameter index out of range");
  const ParamPlan &pp = L->param[p];
  const GroupPlan &gp = L->group[pp.group];
  info->chunk = pp.chunk;
  info->bucket = pp.bucket;
  info->group = pp.group;
  info->bucket_offset = pp.bucket_off;
  info->group_offset = pp.group_off;
  info->ag_byte_offset = gp.byte_off + pp.group_off * dtype_bytes(gp.param_dtype);
  clear_error();
  return FSDP_OK;
}

fsdp_status_t fsdp_layout_bucket(const fsdp_layout_t *L, int32_t b, fsdp_bucket_info_t *info) {
  if (!L || !info) return fail(FSDP_EINVAL, "NULL layout or info");
  if (b < 0 || b >= (int32_t)L->bucket.size()) return fail(FSDP_EINVAL, "bucket index out of range");
  const BucketPlan &bp = L->bucket[b];
  info->reduce_dtype = bp.dtype;
  info->n_params = bp.n_params;
  info->row_elems = bp.S;
  info->bytes = (int64_t)L->W * bp.S * dtype_bytes(bp.dtype);
  clear_error();
  return FSDP_OK;
}

fsdp_status_t fsdp_layout_group(const fsdp_layout_t *L, int32_t g, fsdp_group_info_t *info) {
  if (!L || !info) return fail(FSDP_EINVAL, "NULL layout or info");
  if (g < 0 || g >= (int32_t)L->group.size()) return fail(FSDP_EINVAL, "group index out of range");
  const GroupPlan &gp = L->group[g];
  info->shard_dtype = gp.shard_dtype;
  info->param_dtype = gp.param_dtype;
  info->n_params = gp.n_params;
  info->reserved = 0;
  info->byte_offset = gp.byte_off;
  info->elems = gp.elems;
  info->bytes = gp.elems * dtype_bytes(gp.param_dtype);
  clear_error();
  return FSDP_OK;
}

void fsdp_layout_destroy(fsdp_layout_t *L) {
  if (!L) return;
  device_release(L);
  delete L;
}

const char *fsdp_status_string(fsdp_status_t st) {
  switch (st) {
    case FSDP_OK: return "FSDP_OK";
    case FSDP_EINVAL: return "FSDP_EINVAL";
    case FSDP_ENOMEM: return "FSDP_ENOMEM";
    case FSDP_ECUDA: return "FSDP_ECUDA";
    case FSDP_EUNSUPPORTED: return "FSDP_EUNSUPPORTED";
    case FSDP_ETIMEOUT: return "FSDP_ETIMEOUT";
  }
  return "FSDP_UNKNOWN_STATUS";
}

const char *fsdp_last_error(void) { return g_last_error.c_str(); }

}  // extern "C"
