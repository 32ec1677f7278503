"""Static checks of the prefill kernel's warp-role table (CPU only).

The dequantizing GEMM kernels place their roles on 24 warps by a table (kGemmRoles in
csrc/gemm.cu).  A warp runs on sub-partition (warp index % 4); an epilogue warp may read only
the TMEM lanes of its own sub-partition, so the four epilogue roles must sit on four different
sub-partitions; the MMA issuer, which also allocates TMEM, is warp 1; every role is taken once.
"""
import os
import re

CSRC = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "gguf_block_quantized_gb300",
                    "csrc", "gemm.cu")


def role_table():
    src = open(CSRC).read()
    m = re.search(r"__constant__ uint8_t kGemmRoles\[(\d+)\] = \{([^}]*)\};", src)
    assert m, "role table not found"
    n = int(m.group(1))
    epi0 = 3 + 16  # GEMM_EPI_WARP0 with two teams of 8 dequantizers
    env = {"GEMM_EPI_WARP0": epi0, "GEMM_ROLE_IDLE": 31}
    vals = [eval(v.strip(), {}, env) for v in m.group(2).split(",")]
    assert len(vals) == n
    return vals, epi0


def test_every_role_once_and_the_rest_idle():
    roles, epi0 = role_table()
    taken = [r for r in roles if r != 31]
    assert sorted(taken) == list(range(epi0 + 4))
    assert len(roles) == 24


def test_mma_issuer_is_warp_1_and_its_sub_partition_holds_one_dequantizer():
    roles, epi0 = role_table()
    assert roles[1] == 1  # allocates and frees TMEM as warp 1
    deq_on = [w % 4 for w, r in enumerate(roles) if 3 <= r < epi0]
    assert deq_on.count(1) == 1
    assert len(deq_on) == 16


def test_epilogue_warps_on_four_sub_partitions():
    roles, epi0 = role_table()
    quarters = sorted(w % 4 for w, r in enumerate(roles) if epi0 <= r < epi0 + 4)
    assert quarters == [0, 1, 2, 3]
