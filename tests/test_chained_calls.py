"""Back-to-back decode calls on one stream where a call's input is the previous call's output (a
stacked pair of adapted layers with nothing between them).

The library's kernels let the next kernel on the stream start before they finish, and a decode
call's W tiles normally run before it waits for the kernel before it.  A call whose x overlaps the
outputs of the library's previous call on the stream must wait first.  Here y of an "up"
projection (bf16) is the x of a "down" projection, launched right after it on the same row plan
(no row-plan kernel between the two calls, as in lora_layer_step); the down output is
checked against the oracle computed on the up output the device produced, call after call, and
with an independent x in between (so the W-first path and the waiting path alternate)."""
import numpy as np
import pytest
import torch

import workloads as wl
from harness import bf16_gate, check_close, make_pool, oracle_rows, to_dev_bf16

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)


def test_call_reading_the_previous_calls_output_sees_it_complete():
    import adapter_serving_gb300 as L  # noqa: F401  (the pool comes from the harness)
    n_rows, n_ad = 64, 12
    ranks = np.random.default_rng(3).choice(np.array([8, 16, 32], np.int32), n_ad)
    mods = {"up": (512, 1024), "down": (1024, 512)}
    w = wl.custom("chain", mods, [["up"], ["down"]], n_rows, ranks, 0.5, seed=21,
                  ids=wl.random_ids(n_rows, n_ad, 21, p_base=0.1))
    pool, fac = make_pool(w)
    names = w.module_names()
    iu, idn = names.index("up"), names.index("down")
    Wu, Wd = to_dev_bf16(w.W("up")), to_dev_bf16(w.W("down"))
    ids = torch.from_numpy(w.row_adapters()).cuda()
    x = to_dev_bf16(w.x(0))
    other_x = to_dev_bf16(w.x(1))
    ref_up = oracle_rows(w, "up", 0, factors=fac)
    pool.plan_rows(ids)
    for it in range(4):
        mid = torch.full((n_rows, 1024), float("nan"), dtype=torch.bfloat16, device="cuda")
        y = torch.full((n_rows, 512), float("nan"), dtype=torch.float32, device="cuda")
        spare = torch.empty((n_rows, 512), dtype=torch.float32, device="cuda")
        if it % 2:  # a call with an unrelated x first: the pair then follows a W-first call
            pool.layer_forward_planned([(idn, other_x, Wd, spare)], w.scale)
        pool.layer_forward_planned([(iu, x, Wu, mid)], w.scale)
        pool.layer_forward_planned([(idn, mid, Wd, y)], w.scale)  # x = the previous call's y
        torch.cuda.synchronize()
        mid_bits = mid.view(torch.int16).cpu().numpy().view(np.uint16)
        bad = bf16_gate(mid_bits, ref_up)
        assert bad.size == 0, f"up output, iteration {it}: {len(bad)} outputs outside the bf16 gate"
        ref_down = oracle_rows(w, "down", 1, x_bits=mid_bits, factors=fac)
        check_close(y.cpu().numpy(), ref_down, what=f"down on the up output, iteration {it}")


def test_layer_step_whose_second_stage_reads_the_first_stages_output():
    """The same inside one lora_layer_step call: stage 2's x is stage 1's y."""
    import adapter_serving_gb300 as L  # noqa: F401
    n_rows, n_ad = 48, 10
    ranks = np.random.default_rng(5).choice(np.array([8, 16, 64], np.int32), n_ad)
    mods = {"up": (256, 768), "down": (768, 384)}
    w = wl.custom("chain_step", mods, [["up"], ["down"]], n_rows, ranks, 1.5, seed=23,
                  ids=wl.random_ids(n_rows, n_ad, 23, p_base=0.2))
    pool, fac = make_pool(w)
    names = w.module_names()
    Wu, Wd = to_dev_bf16(w.W("up")), to_dev_bf16(w.W("down"))
    ids = torch.from_numpy(w.row_adapters()).cuda()
    x = to_dev_bf16(w.x(0))
    ref_up = oracle_rows(w, "up", 0, factors=fac)
    for it in range(3):
        mid = torch.full((n_rows, 768), float("nan"), dtype=torch.bfloat16, device="cuda")
        y = torch.full((n_rows, 384), float("nan"), dtype=torch.bfloat16, device="cuda")
        pool.layer_step([[(names.index("up"), x, Wu, mid)], [(names.index("down"), mid, Wd, y)]], ids, w.scale)
        torch.cuda.synchronize()
        mid_bits = mid.view(torch.int16).cpu().numpy().view(np.uint16)
        assert bf16_gate(mid_bits, ref_up).size == 0, f"up output, iteration {it}"
        ref_down = oracle_rows(w, "down", 1, x_bits=mid_bits, factors=fac)
        y_bits = y.view(torch.int16).cpu().numpy().view(np.uint16)
        bad = bf16_gate(y_bits, ref_down)
        assert bad.size == 0, f"down on the up output, iteration {it}: {len(bad)} outputs outside the bf16 gate"
    pool.close()
