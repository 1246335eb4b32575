"""The boundary from a plain C program (CPU only): include/pkv.h compiles as
C11 with strict warnings, and a program linked against libpkv.so runs the
host-side calls (status strings, workspace sizing, the block manager's
prefix hit, fork and copy-on-write) with the results the header documents."""
import os
import shutil
import subprocess

import pytest

import paged_kv_cache_112_gb300 as pkv

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

PROGRAM = r"""
#include <stdio.h>
#include <string.h>
#include "pkv.h"

int main(void) {
  int32_t toks[20], slots[20], slots2[17], table[4], slot, src, dst, i, n, cached;
  int64_t batch[2] = {1, 2};
  int32_t btoks[2] = {5, 6}, bslots[2], blens[2], btables[2][4], bpairs[2][2], sblocks[4], shost[4];
  pkv_bm* bm;
  if (strlen(pkv_status_string(PKV_OK)) == 0) return 1;
  /* one sequence, 1024 tokens, partitions of 512: f32 partial records exist */
  printf("ws %d\n", pkv_decode_workspace_bytes(1, 8, 128, 1024, 512) > 0 ? 1 : 0);
  printf("ws_single %d\n", (int)pkv_decode_workspace_bytes(4, 8, 128, 1024, 0));
  bm = pkv_bm_create(8, 16, 0);
  if (!bm) return 2;
  for (i = 0; i < 20; ++i) toks[i] = 100 + i;
  /* 20 tokens: one full block (cached once written) and a tail of 4 */
  printf("cached1 %d\n", pkv_bm_add_sequence(bm, 1, toks, 20, 0, slots));
  /* the same first 16 tokens: block 0 is a prefix-cache hit, its slots are -1 */
  cached = pkv_bm_add_sequence(bm, 2, toks, 17, 0, slots2);
  printf("cached2 %d first_slot2 %d last_slot2_fresh %d\n", cached, slots2[0], slots2[16] >= 0);
  n = pkv_bm_block_table(bm, 1, table, 4);
  printf("blocks1 %d refcount0 %d\n", n, pkv_bm_block_refcount(bm, table[0]));
  /* a fork shares the tail; the child's append copies it first */
  if (pkv_bm_fork(bm, 1, 3) != PKV_OK) return 3;
  if (pkv_bm_append(bm, 3, 7, &slot, &src, &dst) != PKV_OK) return 4;
  printf("cow_src_is_tail %d cow_dst_fresh %d slot_in_dst %d\n", src == table[1], dst != table[1],
         slot == dst * 16 + 4);
  /* one batched decode step: sequence 1 (tail of 4 shared with nobody now) and 2 (17 tokens) */
  n = pkv_bm_decode_step(bm, batch, btoks, 2, bslots, blens, &btables[0][0], 4, -1, &bpairs[0][0]);
  printf("step_pairs %d lens %d %d pad %d\n", n, blens[0], blens[1], btables[0][3]);
  /* preempt sequence 2 and resume it: its first block is still cached (sequence 1 holds it) */
  if (pkv_bm_swap_out(bm, 2, sblocks, 4) != 2) return 5;
  n = pkv_bm_swap_in_cached(bm, 2, sblocks, shost, 4);
  printf("resume %d from_host %d %d first_shared %d\n", n, shost[0], shost[1], sblocks[0] == table[0]);
  pkv_bm_free_sequence(bm, 1);
  pkv_bm_free_sequence(bm, 2);
  pkv_bm_free_sequence(bm, 3);
  printf("available %d\n", pkv_bm_available_blocks(bm));
  pkv_bm_destroy(bm);
  return 0;
}
"""


def test_header_compiles_as_c11_and_host_calls_run(tmp_path):
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    lib = pkv.library_path()
    if not os.path.exists(lib):
        pytest.skip("libpkv.so is not built")
    src = tmp_path / "consumer.c"
    src.write_text(PROGRAM)
    exe = tmp_path / "consumer"
    libdir = os.path.dirname(lib)
    subprocess.run([cc, "-std=c11", "-Wall", "-Wextra", "-Wpedantic", "-Werror", "-I", os.path.join(ROOT, "include"),
                    str(src), "-o", str(exe), "-L", libdir, "-l:libpkv.so", f"-Wl,-rpath,{libdir}"],
                   check=True, capture_output=True, text=True)
    out = subprocess.run([str(exe)], check=True, capture_output=True, text=True, timeout=60).stdout
    got = dict(line.split(" ", 1) for line in out.strip().splitlines())
    assert got["ws"] == "1"
    assert got["ws_single"] == "0"  # one partition per sequence: no partial records
    assert got["cached1"] == "0"
    assert got["cached2"] == "16 first_slot2 -1 last_slot2_fresh 1"
    assert got["blocks1"] == "2 refcount0 2"
    assert got["cow_src_is_tail"] == "1 cow_dst_fresh 1 slot_in_dst 1"
    assert got["step_pairs"] == "0 lens 21 18 pad -1"
    assert got["resume"] == "2 from_host 0 1 first_shared 1"
    assert got["available"] == "8"
