"""Continuous-batching trace on the GPU: the native scheduler plans each step, the CUDA
path appends the step's tokens and attends over every slot, and the oracle replays the
same appends into its own pool.  Pool bytes are compared bit for bit and attention
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


def _run_trace(tr, steps, check_every):
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
        if len(plan["append_request"]):
            k, v = _step_kv(tr, plan)
            slots = plan["append_slot_mapping"][0]
            pkv.kv_append(pool, U.to_dev(k), U.to_dev(v), U.to_dev(slots), status)
            assert oracle.kv_append(opool, k, v, slots) == 0
        lens = plan["context_lens"]
        q = np.zeros((tr.num_slots, 32, 64), np.uint16)
        if len(plan["decode_slot"]):
            q[plan["decode_slot"]] = tr.step_q(step, plan["decode_slot"])
        bt = np.ascontiguousarray(plan["block_tables"][:, 0, :])
        pkv.paged_decode_attention(pool, out, U.to_dev(q), U.to_dev(bt), bt.shape[1], U.to_dev(lens),
                                   tr.max_context, 0.125, ws, status)
        if step % check_every == 0 or step == steps - 1:
            torch.cuda.synchronize()
            assert int(status.item()) == 0
            np.testing.assert_array_equal(U.bits(pool.view()).reshape(-1), opool.data.reshape(-1))
            ref, err = oracle.paged_decode_attention(opool, q, bt, lens, 0.125, tr.max_context)
            assert err == 0
            U.assert_close(out.cpu().double().numpy(), ref, f"trace step {step}")
            checked += 1
    return sched.stats(), checked


def test_trace_1000_steps_every_tenth():
    tr = configs.trace()
    stats, checked = _run_trace(tr, tr.num_steps, check_every=10)
    assert checked >= 100 and stats["peak_active"] == 32


def test_trace_small_pool_page_reuse():
    tr = configs.trace(seed=186, num_pages=300, num_steps=300)
    stats, checked = _run_trace(tr, tr.num_steps, check_every=10)
    assert stats["admission_waits"] > 0 and stats["peak_pages"] <= 300
