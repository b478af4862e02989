"""Seeded random batches through every kernel path against the fp64 oracle.

Each case draws a head dim (64, 128, 256), page size, layout, group size,
number of kv heads, dtype (bf16, fp16; an FP8 cache for decode plans), an
optional left window, a batch kind (decode; causal or full prefill; mixed
prefill + decode rows) with ragged and empty requests, and an SM count (4
to 152) that forces split decode work, split prefill tiles and persistent
launches with several items per CTA. Every row is compared with the oracle.
V is scaled by 1/4 (exact) so that the output's own rounding stays inside
the budget on rows that see only a few keys."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

from paged_kv_attention_27_gb300 import binding as B  # noqa: E402
from paged_kv_attention_27_gb300 import synth  # noqa: E402

from ._gpu import compare, ensure_built, oracle_parallel, scale_v  # noqa: E402

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    ensure_built()
    B.lib()


def _random_case(seed):
    g = np.random.default_rng(7000 + seed)
    d = int(g.choice([64, 128, 256]))
    P = int(g.choice([16, 32]))
    hkv = int(g.choice([1, 2, 4]))
    grp = int(g.choice([1, 2, 4, 8]))
    kind = str(g.choice(["decode", "decode", "prefill", "mixed"]))
    dtype = "fp16" if g.random() < 0.3 else "bf16"
    layout = synth.NHD if g.random() < 0.5 else synth.HND
    window = int(g.choice([-1, -1, -1, 0, 100, 700, 3000]))
    sms = int(g.choice([4, 8, 30, 152]))
    if kind == "decode":
        batch = int(g.integers(1, 9))
        kv = g.integers(1, 12000, size=batch)
        kv[g.random(batch) < 0.15] = 0
        qo = np.ones(batch, np.int64)
        causal = False
    else:
        batch = int(g.integers(1, 5))
        kv = g.integers(2, 3000, size=batch)
        kv[g.random(batch) < 0.15] = 0
        qo = np.minimum(g.integers(2, 200, size=batch), kv)
        if kind == "mixed":
            qo[(g.random(batch) < 0.5) & (kv > 0)] = 1
        causal = bool(g.random() < 0.8)
        grp = min(grp, 4) if d == 256 else grp
    fp8 = kind == "decode" and g.random() < 0.3
    name = (f"random {seed}: {kind} d{d} P{P} g{grp} hkv{hkv} {dtype}{' fp8' if fp8 else ''} "
            f"w{window} {layout} sms{sms}")
    b = synth.make_batch(name, kv, qo, grp * hkv, hkv, d, P, layout, None, causal, 900 + seed,
                         window_left=window, dtype=dtype, kv_dtype="e4m3" if fp8 else "",
                         kv_scale=1 / 16 if fp8 else 1.0)
    if not fp8:
        scale_v(b)
    mode = B.FI_MODE_DECODE if kind == "decode" else B.FI_MODE_PREFILL
    return b, mode, sms


@pytest.mark.parametrize("seed", range(32))
def test_random_batch_matches_oracle(seed):
    """The device-buffer call against the oracle; the host-buffer call (and,
    for decode plans that fit its scratch, the no-allocation call) bitwise
    the same as the device-buffer call."""
    from paged_kv_attention_27_gb300.device import DeviceBatch
    b, mode, sms = _random_case(seed)
    db = DeviceBatch(b, mode=mode, sms=sms)
    out, lse = db.run()
    torch.cuda.synchronize()
    if int(b.qo_lens.sum()) == 0:      # every request empty: the call ran nothing
        return
    assert db.status() == B.FI_OK, b.name
    out, lse = out.clone(), lse.clone()
    ref_o, ref_l = oracle_parallel(b)
    compare(out, lse, ref_o, ref_l, what=b.name)
    same = lambda o, l: (torch.equal(o.view(torch.int16).cpu(), out.view(torch.int16).cpu()) and
                         torch.equal(l.cpu(), lse.cpu()))
    out_h, lse_h = db.run_host()
    assert same(out_h, lse_h), f"{b.name}: host-buffer call differs"
    if mode == B.FI_MODE_DECODE and B.fi_plan_get_info(db.plan)["workspace_bytes"] <= 16 << 20:
        o2 = torch.full_like(out, float("nan"))
        l2 = torch.full_like(lse, float("nan"))
        B.fi_batch_decode_paged_noalloc(db.plan, db.q, db.k, db.v, B.LAYOUTS[b.layout], 0,
                                        b.num_pages, db.page_indptr, db.page_indices,
                                        db.last_page_len, b.sm_scale, b.k_scale, b.v_scale, o2,
                                        l2, k_head_scale=db.k_head_scale,
                                        v_head_scale=db.v_head_scale)
        torch.cuda.synchronize()
        assert same(o2, l2), f"{b.name}: no-allocation call differs"
