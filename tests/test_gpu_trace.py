"""Continuous-batching trace on the GPU: the native scheduler plans each step, the CUDA
path appends the step's tokens and attends over every slot, and the oracle replays the
same appends into its own pool (the GPU side either appends every token and then attends, or
appends the admitted prompts and runs the fused decode step, which appends each decoding
slot's new token itself).  Pool bytes are compared bit for bit and attention
against the oracle at every tenth step (32 slots, 1 layer, prompts U[16, 512], budgets
U[1, 512], 4096-page pool; plus a small pool where requests wait and pages are reused).
"""
import numpy as np
import pytest
import torch

import oracle
from tests import gpu_util as U
from workloads import configs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def _step_kv(tr, plan):
    """K/V of the plan's appended tokens, in plan order (runs of consecutive positions per request)."""
    reqs, pos = plan["append_request"], plan["append_position"]
    ks, vs = [], []
    i = 0
    while i < len(reqs):
        j = i
        while j + 1 < len(reqs) and reqs[j + 1] == reqs[i] and pos[j + 1] == pos[j] + 1:
            j += 1
        k, v = tr.request_kv(int(reqs[i]), int(pos[i]), int(pos[j]) + 1)
        ks.append(k)
        vs.append(v)
        i = j + 1
    return np.concatenate(ks), np.concatenate(vs)


def _run_trace(tr, steps, check_every, fused=False):
    import paged_kv_cache_180_gb300 as pkv
    sched = pkv.Scheduler(tr.num_pages, 1, 16, tr.max_context, tr.num_slots, tr.free_order)
    for rid in range(tr.num_requests):
        sched.submit(rid, int(tr.prompt_lens[rid]), int(tr.new_budgets[rid]))
    pool = pkv.KVPool(tr.num_pages, device=U.dev())
    pool.buffer.view(torch.int16).fill_(-1)
    opool = oracle.Pool(tr.num_pages)
    status = torch.zeros(1, dtype=torch.int32, device=U.dev())
    ws = pkv.decode_workspace(tr.num_slots, device=U.dev())
    out = torch.empty(tr.num_slots, 32, 64, dtype=torch.float32, device=U.dev())
    checked = 0
    for step in range(steps):
        plan = sched.step()
        lens = plan["context_lens"]
        q = np.zeros((tr.num_slots, 32, 64), np.uint16)
        dec = plan["decode_slot"]
        if len(dec):
            q[dec] = tr.step_q(step, dec)
        bt = np.ascontiguousarray(plan["block_tables"][:, 0, :])
        n_app = len(plan["append_request"])
        if n_app:
            k, v = _step_kv(tr, plan)
            slots = plan["append_slot_mapping"][0]
            assert oracle.kv_append(opool, k, v, slots) == 0
        if not fused:
            if n_app:
                pkv.kv_append(pool, U.to_dev(k), U.to_dev(v), U.to_dev(slots), status)
            pkv.paged_decode_attention(pool, out, U.to_dev(q), U.to_dev(bt), bt.shape[1], U.to_dev(lens),
                                       tr.max_context, 0.125, ws, status)
        else:
            # admitted prompts (listed first) through kv_append; each decoding slot's new token
            # (listed last, slots ascending) through the fused step, slot -1 where none
            n_pr = n_app - len(dec)
            if n_pr:
                pkv.kv_append(pool, U.to_dev(k[:n_pr]), U.to_dev(v[:n_pr]), U.to_dev(slots[:n_pr]), status)
            kn = np.zeros((tr.num_slots, 8, 64), np.uint16)
            vn = np.zeros((tr.num_slots, 8, 64), np.uint16)
            sn = np.full(tr.num_slots, -1, np.int32)
            if len(dec):
                kn[dec], vn[dec], sn[dec] = k[n_pr:], v[n_pr:], slots[n_pr:]
            pkv.decode_step(pool, U.to_dev(kn), U.to_dev(vn), U.to_dev(sn), out, U.to_dev(q), U.to_dev(bt),
                            bt.shape[1], U.to_dev(lens), tr.max_context, 0.125, ws, status)
        if step % check_every == 0 or step == steps - 1:
            torch.cuda.synchronize()
            assert int(status.item()) == 0
            np.testing.assert_array_equal(U.bits(pool.view()).reshape(-1), opool.data.reshape(-1))
            ref, err = oracle.paged_decode_attention(opool, q, bt, lens, 0.125, tr.max_context)
            assert err == 0
            U.assert_close(out.cpu().double().numpy(), ref, f"trace step {step}")
            checked += 1
    return sched.stats(), checked


@pytest.mark.parametrize("fused", [False, True], ids=["append_then_attend", "fused_decode_step"])
def test_trace_1000_steps_every_tenth(fused):
    tr = configs.trace()
    stats, checked = _run_trace(tr, tr.num_steps, check_every=10, fused=fused)
    assert checked >= 100 and stats["peak_active"] == 32


def test_trace_small_pool_page_reuse():
    tr = configs.trace(seed=186, num_pages=300, num_steps=300)
    stats, checked = _run_trace(tr, tr.num_steps, check_every=10)
    assert stats["admission_waits"] > 0 and stats["peak_pages"] <= 300
