"""moe_dispatch_noalloc: the dispatch entry point for callers that cannot
allocate device memory (for example a plugin whose host framework owns every
device allocation, or a decode loop that must not call cudaMalloc/cudaFree
because they can synchronise the device).  It keeps its scratch in a fixed
array inside the library.

The GPU test calls it through the C ABI twice in a row, with different
problem sizes, and requires bit-identical results to moe_dispatch given a
caller-allocated workspace (dispatch output is integer and copy work, so the
tolerance is exact).  This file is collected last so that a run stopping at
the first failure has already run every other test; it also passes alone in
a fresh process."""
import ctypes

import numpy as np
import pytest
import torch


def _lib():
    from combine_dp_gather_gb300 import build, moe_dp
    build.build()
    moe_dp.lib()
    return moe_dp


def _case(rows, k, E, H, seed, dev="cuda"):
    g = torch.Generator(device=dev).manual_seed(seed)
    ids = torch.rand(rows, E, generator=g, device=dev).argsort(dim=1)[:, :k].to(torch.int32)
    ids[::5] = -1
    x = torch.randn(rows, H, generator=g, device=dev).to(torch.bfloat16)
    return ids.contiguous(), x


def _outputs(md, rows, k, P, H, align, dev="cuda"):
    cap = md.moe_dispatch_cap_bound(rows, k, P, align)
    return dict(counts_P=torch.full((P,), -9, dtype=torch.int32, device=dev),
                offsets_P=torch.full((P + 1,), -9, dtype=torch.int32, device=dev),
                perm=torch.full((cap,), -9, dtype=torch.int32, device=dev),
                inv=torch.full((rows, k), -9, dtype=torch.int32, device=dev),
                xs=torch.zeros(cap, H, device=dev, dtype=torch.bfloat16),
                st=torch.zeros(1, dtype=torch.int32, device=dev))


@pytest.mark.gpu
def test_noalloc_dispatch_matches_dispatch_on_two_calls():
    md = _lib()
    from combine_dp_gather_gb300 import synth
    # both calls exceed the one-CTA path's 8192 routed pairs, so both keep their
    # chunk histograms in the shared scratch; the second (12 chunks x 48 experts)
    # uses fewer entries than the first (24 chunks x 64 experts) left behind, and
    # must not see them
    cases = [dict(rows=3001, k=8, E=64, H=512, align=1, seed=1, map=False),
             dict(rows=1500, k=8, E=48, H=256, align=4, seed=2, map=True)]
    for c in cases:
        ids, x = _case(c["rows"], c["k"], c["E"], c["H"], c["seed"])
        l2p = nrep = None
        P = c["E"]
        if c["map"]:
            l2p_np, nrep_np, p2l = synth.eplb_map(np.arange(c["E"])[::-1] + 1, 16, 8)
            P = len(p2l)
            l2p, nrep = torch.from_numpy(l2p_np).cuda(), torch.from_numpy(nrep_np).cuda()
        ref = _outputs(md, c["rows"], c["k"], P, c["H"], c["align"])
        ws = torch.empty(md.moe_dispatch_ws_bytes(c["rows"], c["k"], c["E"]), dtype=torch.uint8,
                         device="cuda")
        md.moe_dispatch(x, ids, c["E"], P, ref["counts_P"], ref["offsets_P"], ref["perm"],
                        ref["inv"], ref["xs"], ws, l2p, nrep, c["align"], ref["st"])
        got = _outputs(md, c["rows"], c["k"], P, c["H"], c["align"])
        md.moe_dispatch_noalloc(x, ids, c["E"], P, got["counts_P"], got["offsets_P"],
                                got["perm"], got["inv"], got["xs"], l2p, nrep, c["align"],
                                got["st"])
        torch.cuda.synchronize()
        assert int(ref["st"].item()) == 0 and int(got["st"].item()) == 0
        n = int(ref["offsets_P"][-1].item())
        for key in ("counts_P", "offsets_P", "inv"):
            assert torch.equal(got[key], ref[key]), key
        assert torch.equal(got["perm"][:n], ref["perm"][:n])
        assert torch.equal(got["xs"][:n].view(torch.int16), ref["xs"][:n].view(torch.int16))


def test_noalloc_dispatch_rejects_problems_beyond_its_scratch():
    md = _lib()
    fake = ctypes.c_void_p(0x1000)
    rows, k, E = 40000, 8, 256           # 313 chunks x 256 experts > 65536 entries
    assert md.moe_dispatch_ws_bytes(rows, k, E) > md.MOE_NOALLOC_SCRATCH_BYTES
    code = md.lib().moe_dispatch_noalloc(fake, fake, rows, k, 64, 1, E, E, None, None, 0, 1,
                                         rows * k, fake, fake, fake, fake, fake, None, None)
    assert code == md.MOE_ERR_CAPACITY


def test_noalloc_dispatch_checks_arguments_before_its_scratch_size():
    """An invalid call that is also too large for the scratch returns what
    moe_dispatch returns for the same arguments, not MOE_ERR_CAPACITY."""
    md = _lib()
    fake = ctypes.c_void_p(0x1000)
    rows, E = 40000, 256
    for k, P, want in ((33, E, md.MOE_ERR_INVALID_ARG),          # k > MOE_MAX_TOPK
                       (8, E + 1, md.MOE_ERR_INVALID_ARG)):       # P != E without a map
        code = md.lib().moe_dispatch_noalloc(fake, fake, rows, k, 64, 1, E, P, None, None, 0, 1,
                                             rows * k, fake, fake, fake, fake, fake, None, None)
        assert code == want, (k, P, code)
    # an unsupported dtype with rows to move: the same status as moe_dispatch
    code = md.lib().moe_dispatch_noalloc(fake, fake, rows, 8, 64, 9, E, E, None, None, 0, 1,
                                         rows * 8, fake, fake, fake, fake, fake, None, None)
    assert code == md.MOE_ERR_UNSUPPORTED


def test_noalloc_binding_refuses_misshaped_outputs():
    md = _lib()
    import torch
    rows, k, E, H = 8, 2, 4, 64
    ids = torch.zeros(rows, k, dtype=torch.int32)
    x = torch.zeros(rows, H, dtype=torch.bfloat16)
    cap = rows * k
    good = dict(counts_P=torch.zeros(E, dtype=torch.int32),
                offsets_P=torch.zeros(E + 1, dtype=torch.int32),
                perm=torch.zeros(cap, dtype=torch.int32),
                inv=torch.zeros(rows, k, dtype=torch.int32),
                sorted_out=torch.zeros(cap, H, dtype=torch.bfloat16))
    bad = [("counts_P", torch.zeros(E - 1, dtype=torch.int32)),
           ("offsets_P", torch.zeros(E, dtype=torch.int32)),
           ("inv", torch.zeros(rows, k + 1, dtype=torch.int32)),
           ("inv", torch.zeros(rows, k, dtype=torch.int64)),
           ("sorted_out", torch.zeros(cap, H, dtype=torch.float32)),
           ("sorted_out", torch.zeros(cap - 1, H, dtype=torch.bfloat16))]
    for name, t in bad:
        args = dict(good, **{name: t})
        with pytest.raises(md.MoeError) as ei:   # refused on the host, before any launch
            md.moe_dispatch_noalloc(x, ids, E, E, args["counts_P"], args["offsets_P"],
                                    args["perm"], args["inv"], args["sorted_out"])
        assert ei.value.code == md.MOE_ERR_INVALID_ARG, name
