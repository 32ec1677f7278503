"""The prefill product's tile schedule (host logic, CPU only): syn_debug_prefill_plan.

The product computes 128 x BN tiles (BN = n_tok rounded up to 16, at most 256) over K in
256-wide super-steps.  Tiles that fill whole waves of the SMs run whole; the tiles of a last,
partial wave are split along K S ways (adding into a zeroed Y), or, for long K (at least 32
super-steps), shared stream-K; products with fewer tiles than SMs and long K run stream-K
throughout.  The expected schedules below are the planner's choices on 152 SMs for the
Llama-8B shapes (the benchmark's), which the GPU timings of each alternative supported.
"""
import ctypes
import random

import pytest

from gguf_block_quantized_gb300 import syn


def plan(n_out, n_in, n_tok, sms=152):
    out = (ctypes.c_int * 4)()
    assert syn.syn_debug_prefill_plan(n_out, n_in, n_tok, sms, out) == syn.OK
    return {"S": out[0], "m_full": out[1], "streamk": bool(out[2]), "tiles": out[3]}


@pytest.mark.parametrize("shape,n_tok,want", [
    ((4096, 14336), 2048, {"S": 1, "m_full": 19, "streamk": True, "tiles": 256}),   # FFN down: stream-K tail
    ((4096, 14336), 512, {"S": 1, "m_full": 0, "streamk": True, "tiles": 64}),      # FFN down: stream-K
    ((14336, 4096), 512, {"S": 2, "m_full": 76, "streamk": False, "tiles": 224}),   # FFN up: split tail
    ((14336, 4096), 2048, {"S": 1, "m_full": 112, "streamk": False, "tiles": 896}),  # FFN up: whole tiles
    ((4096, 4096), 2048, {"S": 4, "m_full": 19, "streamk": False, "tiles": 256}),   # q/o: split tail
    ((1024, 4096), 2048, {"S": 2, "m_full": 0, "streamk": False, "tiles": 64}),     # k/v: split
])
def test_llama8b_schedules(shape, n_tok, want):
    got = plan(shape[0], shape[1], n_tok)
    if want["S"] == 1 and not want["streamk"]:
        got["m_full"] = want["m_full"]  # whole tiles only: m_full is not used
    assert got == want


def test_schedule_invariants_on_random_shapes():
    rng = random.Random(11)
    for _ in range(400):
        n_out = rng.randint(1, 40000)
        n_in = 256 * rng.randint(1, 80)
        n_tok = rng.randint(9, 5000)
        sms = rng.choice([1, 7, 8, 64, 152])
        p = plan(n_out, n_in, n_tok, sms)
        bn = min(256, (n_tok + 15) // 16 * 16)
        n_m, n_n, n_super = -(-n_out // 128), -(-n_tok // bn), -(-n_in // 256)
        assert p["tiles"] == n_m * n_n
        assert 1 <= p["S"] <= 16 and 0 <= p["m_full"] <= n_m
        if p["streamk"]:
            assert p["S"] == 1 and n_super >= 32
            # the whole tiles before the shared ones fill whole waves, or there are none
            assert p["m_full"] * n_n <= (p["tiles"] // sms) * sms
        if p["S"] > 1:
            assert n_super // p["S"] >= 2  # every split keeps at least two super-steps
            assert p["m_full"] < n_m


def test_argument_checks():
    out = (ctypes.c_int * 4)()
    assert syn.syn_debug_prefill_plan(0, 256, 16, 152, out) == syn.ERR_SHAPE
    assert syn.syn_debug_prefill_plan(128, 256, 16, 0, out) == syn.ERR_SHAPE
    assert syn.syn_debug_prefill_plan(128, 256, 16, 152, None) == syn.ERR_NULL
