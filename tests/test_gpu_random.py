"""Seeded random batches on the GPU against the oracle, element by element.

Each case draws a batch shape the hand-written tests do not pin down: the number of
sequences, a length mix (uniform, mostly short with a few long ones, all equal, or with
zero lengths), the split (automatic, or a caller-fixed CTA count), and the entry point
(attention after a bulk append, or the fused append + attention step).  Prefill cases
draw per-sequence query chunks (full prompts, chunks after a cached prefix, single
queries) and lengths that are not multiples of the 32-token tile or the 16-token page.
Tolerance |gpu - oracle| <= 1e-3 + 1e-2 |oracle|; the pool bytes after the fused step are
compared bit for bit.
"""
import numpy as np
import pytest
import torch

import oracle
from tests import gpu_util as U
from workloads import configs, rng

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def _lengths(r, n, mix):
    if mix == "uniform":
        return r.integers(1, 2049, n)
    if mix == "short_and_long":
        lens = r.integers(1, 64, n)
        lens[r.random(n) < 0.1] = r.integers(1024, 2049)
        return lens
    if mix == "equal":
        return np.full(n, int(r.integers(1, 2049)))
    lens = r.integers(0, 2049, n)           # "with_zeros": some sequences have no tokens at all
    lens[r.random(n) < 0.2] = 0
    return lens


CASES = [(seed, mix) for seed in range(12) for mix in ("uniform", "short_and_long", "equal", "with_zeros")][::3]


@pytest.mark.parametrize("seed,mix", CASES, ids=[f"{s}-{m}" for s, m in CASES])
def test_random_decode_batches(seed, mix):
    import paged_kv_cache_180_gb300 as pkv
    r = np.random.default_rng(7000 + seed)
    n = int(r.choice([1, 2, 3, 7, 31, 64, 150, 305]))
    lens = _lengths(r, n, mix)
    wl = configs.custom(7000 + seed, lens.tolist(), num_pages=None, name=f"random-{seed}-{mix}")
    fused = bool(r.integers(0, 2))
    ctas = int(r.choice([0, 0, 1, 5, 97, 304, 1024]))
    d = U.DeviceDecode(wl)
    if fused:
        # the pool holds every token but each sequence's last; the fused step appends it
        from workloads import torch_gen
        k, v, slots = torch_gen.workload_kv(wl, 0, U.dev(), upto_offset=1)
        if slots.numel():
            pkv.kv_append(d.pool, k, v, slots, d.status)
        kn = np.zeros((n, 8, 64), np.uint16)
        vn = np.zeros((n, 8, 64), np.uint16)
        sn = np.full(n, -1, np.int32)
        live = [s for s in range(n) if lens[s] > 0]
        if live:
            kd, vd, sd = wl.decode_tokens(0)
            kn[live], vn[live], sn[live] = kd, vd, sd
        pkv.decode_step(d.pool, U.to_dev(kn), U.to_dev(vn), U.to_dev(sn), d.out, d.q(0), d.bt.view(-1),
                        wl.max_blocks, d.lens, wl.max_context, wl.scale, d.ws, d.status)
        out = d.out
    else:
        d.append_all()
        out = d.attend(0, num_ctas=ctas)
    got = out.cpu().double().numpy()
    assert d.status_value() == 0
    ref, err = U.oracle_decode_threaded(wl)
    assert err == 0
    U.assert_close(got, ref, f"{wl.name} (n={n}, fused={fused}, ctas={ctas})")
    if fused:
        opool = oracle.Pool(wl.num_pages)
        k, v, slots = wl.kv_all(0)
        oracle.kv_append(opool, k, v, slots)
        np.testing.assert_array_equal(U.bits(d.pool.view()).reshape(-1), opool.data.reshape(-1))


@pytest.mark.parametrize("seed", range(10))
def test_random_prefill_batches(seed):
    import paged_kv_cache_180_gb300 as pkv
    r = np.random.default_rng(8000 + seed)
    n = int(r.choice([1, 2, 5, 9, 16]))
    lens = r.integers(1, 700, n)
    nq = []
    for c in lens:
        kind = r.integers(0, 3)
        nq.append(int(c) if kind == 0 else (1 if kind == 1 else int(r.integers(1, c + 1))))
    wl = configs.custom(8000 + seed, lens.tolist(), name=f"prefill-random-{seed}")
    d = U.DeviceDecode(wl)
    d.append_all()
    qs = np.concatenate([[0], np.cumsum(nq)]).astype(np.int32)
    total = int(qs[-1])
    qbits = rng.normal_bf16(rng.stream_key(8000 + seed, "pf-q"), 0, total * 32 * 64).reshape(total, 32, 64)
    out = torch.full((total, 32, 64), float("nan"), dtype=torch.float32, device=U.dev())
    bt_host = np.ascontiguousarray(wl.block_tables[:, 0, :])
    pkv.paged_prefill_attention(d.pool, out, U.to_dev(qbits), U.to_dev(qs), U.to_dev(bt_host), bt_host.shape[1],
                                d.lens, max(nq), wl.max_context, wl.scale, d.status)
    assert d.status_value() == 0
    opool = oracle.Pool(wl.num_pages)
    k, v, slots = wl.kv_all(0)
    oracle.kv_append(opool, k, v, slots)
    ref, err = oracle.paged_prefill_attention(opool, qbits, qs, bt_host, wl.context_lens, wl.scale, wl.max_context)
    assert err == 0
    U.assert_close(out.cpu().double().numpy(), ref, f"{wl.name} (n={n})")
