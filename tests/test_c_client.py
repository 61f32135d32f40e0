"""The boundary as a C program sees it, without a GPU.

A small C99 client is compiled with gcc in strict mode (-std=c99 -pedantic
-Wall -Wextra -Werror) against include/fsdp_pack.h alone -- no CUDA header --
and linked to the built library.  It plans the two-block model of Linear(6, 6)
units from "The unit you wrapped" (auto_wrap_policy section) on the host at
W = 4, as one group of all four layers and as one group per layer, and prints
every queried size and offset.  The printed values must equal the oracle's
plan, and the per-rank counts must be the page's: 36 elements for the single
unit and 9 per Linear.  It also checks the documented refusals (W < 1, an
unknown dtype, a NULL output), each with FSDP_EINVAL and a message, and that
an empty group plans.
"""
import os
import shutil
import subprocess

import pytest

import oracle
from fsdp2_gradient_packing_gb300 import _build
from fsdp2_gradient_packing_gb300 import workloads as wl

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CLIENT = r"""
#include <stdio.h>
#include <string.h>
#include "fsdp_pack.h"

static int plan_and_print(const fsdp_param_desc_t *d, int32_t n, int32_t W, const char *tag) {
  fsdp_layout_t *L = NULL;
  fsdp_layout_info_t info;
  int32_t p, b, g;
  if (fsdp_plan_layout_host(d, n, W, &L) != FSDP_OK) return 1;
  if (fsdp_layout_query(L, &info) != FSDP_OK) return 2;
  printf("%s layout %d %d %d %d %lld %lld %d %d\n", tag, (int)info.world_size, (int)info.n_params,
         (int)info.n_buckets, (int)info.n_groups, (long long)info.ag_bytes, (long long)info.total_numel,
         (int)info.device, (int)info.has_device_table);
  for (p = 0; p < info.n_params; ++p) {
    fsdp_param_info_t pi;
    if (fsdp_layout_param(L, p, &pi) != FSDP_OK) return 3;
    printf("%s param %d %lld %d %lld %d %lld %lld\n", tag, (int)p, (long long)pi.chunk, (int)pi.bucket,
           (long long)pi.bucket_offset, (int)pi.group, (long long)pi.group_offset,
           (long long)pi.ag_byte_offset);
  }
  for (b = 0; b < info.n_buckets; ++b) {
    fsdp_bucket_info_t bi;
    if (fsdp_layout_bucket(L, b, &bi) != FSDP_OK) return 4;
    printf("%s bucket %d %d %lld %lld\n", tag, (int)b, (int)bi.reduce_dtype, (long long)bi.row_elems,
           (long long)bi.bytes);
  }
  for (g = 0; g < info.n_groups; ++g) {
    fsdp_group_info_t gi;
    if (fsdp_layout_group(L, g, &gi) != FSDP_OK) return 5;
    printf("%s group %d %d %d %lld %lld\n", tag, (int)g, (int)gi.shard_dtype, (int)gi.param_dtype,
           (long long)gi.byte_offset, (long long)gi.elems);
  }
  if (fsdp_layout_param(L, info.n_params, NULL) != FSDP_EINVAL) return 6;
  fsdp_layout_destroy(L);
  return 0;
}

int main(void) {
  fsdp_param_desc_t d[4];
  fsdp_layout_t *L = NULL;
  int k, rc;
  for (k = 0; k < 4; ++k) {
    d[k].numel = 36;
    d[k].grad_dtype = k < 2 ? FSDP_DTYPE_F32 : FSDP_DTYPE_BF16;
    d[k].reduce_dtype = FSDP_DTYPE_F32;
    d[k].shard_dtype = FSDP_DTYPE_F32;
    d[k].param_dtype = FSDP_DTYPE_BF16;
  }
  if ((rc = plan_and_print(d, 4, 4, "model")) != 0) return 10 + rc;
  for (k = 0; k < 4; ++k) {
    char tag[16];
    sprintf(tag, "linear%d", k);
    if ((rc = plan_and_print(d + k, 1, 4, tag)) != 0) return 20 + rc;
  }
  if ((rc = plan_and_print(NULL, 0, 4, "empty")) != 0) return 30 + rc;

  if (fsdp_plan_layout_host(d, 4, 0, &L) != FSDP_EINVAL || L != NULL) return 40;
  if (strlen(fsdp_last_error()) == 0) return 41;
  printf("refused W=0: %s\n", fsdp_last_error());
  d[1].param_dtype = 7;
  if (fsdp_plan_layout_host(d, 4, 4, &L) != FSDP_EINVAL || L != NULL) return 42;
  printf("refused dtype: %s\n", fsdp_last_error());
  d[1].param_dtype = FSDP_DTYPE_BF16;
  if (fsdp_plan_layout_host(d, 4, 4, NULL) != FSDP_EINVAL) return 43;
  if (strcmp(fsdp_status_string(FSDP_EINVAL), fsdp_status_string(FSDP_OK)) == 0) return 44;
  printf("ok\n");
  return 0;
}
"""


@pytest.fixture(scope="module")
def client(tmp_path_factory):
    if shutil.which("gcc") is None:
        pytest.skip("gcc not found")
    lib = _build.build()
    d = tmp_path_factory.mktemp("c_client")
    src, exe = d / "client.c", d / "client"
    src.write_text(CLIENT)
    libdir = os.path.dirname(lib)
    cmd = ["gcc", "-std=c99", "-pedantic", "-Wall", "-Wextra", "-Werror", "-I", os.path.join(ROOT, "include"),
           str(src), "-o", str(exe), "-L", libdir, "-l:" + os.path.basename(lib), "-Wl,-rpath," + libdir]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=60)
    assert r.returncode == 0, (r.returncode, r.stdout, r.stderr)
    return r.stdout.splitlines()


def _records(lines, tag, kind):
    return [[int(x) for x in ln.split()[2:]] for ln in lines if ln.split()[:2] == [tag, kind]]


def _expected(specs, W):
    pl = oracle.plan(oracle.params_from_specs(specs), W)
    layout = [W, len(specs), len(pl.bucket_dtype), len(pl.group_pair), pl.S_ag, sum(s.numel for s in specs), -1, 0]
    params = [[p, pl.chunk[p], pl.bucket_of[p], pl.bucket_off[p], pl.group_of[p], pl.group_elem_off[p],
               pl.group_byte_off[pl.group_of[p]] + pl.group_elem_off[p] * (2 if pl.group_pair[pl.group_of[p]][1]
                                                                           == oracle.BF16 else 4)]
              for p in range(len(specs))]
    buckets = [[b, pl.bucket_dtype[b], pl.bucket_S[b], W * pl.bucket_S[b] * (4 if pl.bucket_dtype[b] == oracle.F32
                                                                              else 2)]
               for b in range(len(pl.bucket_dtype))]
    groups = [[g, pl.group_pair[g][0], pl.group_pair[g][1], pl.group_byte_off[g], pl.group_elems[g]]
              for g in range(len(pl.group_pair))]
    return layout, params, buckets, groups


def test_c_client_plans_as_the_oracle_does(client):
    work = wl.tiny_two_blocks(W=4, grouping="model")
    cases = [("model", list(work.groups[0]))] + [(f"linear{k}", [work.groups[0][k]]) for k in range(4)]
    for tag, specs in cases:
        layout, params, buckets, groups = _expected(specs, 4)
        assert _records(client, tag, "layout") == [layout], tag
        assert _records(client, tag, "param") == params, tag
        assert _records(client, tag, "bucket") == buckets, tag
        assert _records(client, tag, "group") == groups, tag
    assert _records(client, "empty", "layout") == [[4, 0, 0, 0, 0, 0, -1, 0]]
    assert client[-1] == "ok"


def test_c_client_prints_the_page_counts(client):
    """One unit of all four Linear(6, 6) layers: 36 elements per rank; one
    unit per Linear: 9 ("The unit you wrapped", auto_wrap_policy section)."""
    assert [r[2] for r in _records(client, "model", "bucket")] == [36]
    for k in range(4):
        assert [r[2] for r in _records(client, f"linear{k}", "bucket")] == [9]
        assert [r[1] for r in _records(client, f"linear{k}", "param")] == [9]
