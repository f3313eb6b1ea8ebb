"""The expert residency bank on the GPU: every banked forward gives the resident forward's bits,
the bank's state after each forward equals the oracle's bank plan bit for bit, and the first
forward of each case matches the oracle's layer output."""
import dataclasses

import numpy as np
import pytest

from routed_moe_fp4_gb300 import synthetic as S
from tests import parity as P

pytestmark = pytest.mark.gpu


def _run_bank(oracle, name, slots, Ts, check_tokens=8, copy_blocks=None, seed_batches=1):
    import torch
    from oracle.oracle import BankState, bank_plan
    from routed_moe_fp4_gb300 import colimoe as cm
    base = S.make_inputs(name)
    wl = base.workload
    Tm = max(Ts)
    layer = cm.MoELayer(base, max_tokens=Tm)
    layer.set_ffn_path(cm.COLI_FFN_GEMM_MXF4)
    bank = cm.ExpertBank(layer, slots, cm.HostExperts(base.experts))
    if copy_blocks:
        bank.set_copy_blocks(copy_blocks)
    st = BankState(wl.E, slots)
    for n, T in enumerate(Ts):
        xb = S.x_batch(0, wl.name, seed_batches + n, T, wl.H)
        x = torch.from_numpy(xb.view(np.int16)).cuda()
        ref = torch.empty((T, wl.H), dtype=torch.int16, device="cuda")
        got = torch.full((T, wl.H), -1, dtype=torch.int16, device="cuda")
        layer.forward(x, ref)
        bank.forward(x, got)
        torch.cuda.synchronize()
        assert layer.device_error() == 0
        assert torch.equal(ref, got), f"forward {n} (T={T}): banked output differs from the resident one"
        routing = layer.routing(T)
        rnd, slot, cop = bank_plan(oracle, st, routing["cnt"], T, wl.top_k)
        dev = bank.state()
        for key in ("slot_of", "expert_in", "usage", "last_use", "stats"):
            assert np.array_equal(dev[key], getattr(st, key)), f"forward {n} (T={T}): bank {key} differs"
        if n == 0 and check_tokens:
            inputs = dataclasses.replace(base, x=xb, workload=dataclasses.replace(wl, T=T))
            toks = P.sample_tokens(routing, T, min(check_tokens, T))
            rep = P.check(oracle, inputs, got.cpu().numpy().view(np.uint16), routing, tokens=toks)
            assert rep.ok, rep
    stats = bank.state()["stats"]
    bank.close()
    layer.close()
    return stats


def test_bank_decode_cache(oracle):
    """Decode forwards (T 8, top-8, 256 experts) over a bank of 64 slots: cache forwards, resident
    experts in place, the others copied while they compute."""
    stats = _run_bank(oracle, "decode", 64, [8] * 6)
    assert stats[0] == 6 and stats[2] > 0


def test_bank_transient_rounds(oracle):
    """T 16 and 48 over 64 slots: 128 and 384 routed slots exceed the bank, so transient forwards in
    groups of 32 (4 and 8 rounds), each group's copies overlapping the previous group's GEMMs."""
    _run_bank(oracle, "decode", 64, [16, 48, 16], check_tokens=6)


def test_bank_mixed_sequence(oracle):
    """Cache and transient forwards in turn; the bank state carries across them."""
    _run_bank(oracle, "decode", 48, [8, 24, 4, 8, 2], check_tokens=4)


def test_bank_prefill_small_bank(oracle):
    """A 512-token prefill over a bank of 32 slots: 16 rounds of 16 experts."""
    _run_bank(oracle, "prefill", 32, [512], check_tokens=6)


@pytest.mark.parametrize("slots", [2, 3, 8])
def test_bank_tiny_edges(oracle, slots):
    """8 experts, top-2: two slots (one expert per round), an odd slot count, and a bank as large
    as the expert set."""
    _run_bank(oracle, "tiny", slots, [4, 1, 4, 3], check_tokens=4)


def test_bank_copy_blocks(oracle):
    """The result does not depend on how many blocks copy while another round computes."""
    _run_bank(oracle, "decode", 64, [8, 16], check_tokens=0, copy_blocks=1)
    _run_bank(oracle, "decode", 64, [8, 16], check_tokens=0, copy_blocks=64)


def test_bank_graph_capture():
    """A banked forward captured in a CUDA graph replays to the eager forward's bits."""
    import torch
    from routed_moe_fp4_gb300 import colimoe as cm
    base = S.make_inputs("decode")
    wl = base.workload
    stream = torch.cuda.Stream()
    layer = cm.MoELayer(base, stream=stream)
    bank = cm.ExpertBank(layer, 64, cm.HostExperts(base.experts))
    x = torch.from_numpy(S.x_batch(0, wl.name, 1, wl.T, wl.H).view(np.int16)).cuda()
    eager = torch.empty((wl.T, wl.H), dtype=torch.int16, device="cuda")
    out = torch.empty_like(eager)
    with torch.cuda.stream(stream):
        bank.forward(x, eager)
    stream.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        bank.forward(x, out)
    for _ in range(3):
        out.fill_(0)
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(out, eager)
    assert layer.device_error() == 0
    bank.close()
    layer.close()


def test_bank_rejects_bad_arguments():
    import torch
    from routed_moe_fp4_gb300 import colimoe as cm
    base = S.make_inputs("tiny")
    layer = cm.MoELayer(base)
    host = cm.HostExperts(base.experts)
    for slots in (1, base.workload.E + 1):
        with pytest.raises(cm.ColiError):
            cm.ExpertBank(layer, slots, host)
    pageable = cm.coli_mxfp4_experts(*[a.ctypes.data for a in (base.experts.gate_up_codes,
                                                                base.experts.gate_up_scales,
                                                                base.experts.down_codes,
                                                                base.experts.down_scales)])
    with pytest.raises(cm.ColiError):
        cm.coli_bank_create(layer.h, 4, pageable)
    layer.close()
    torch.cuda.synchronize()
