"""Randomised checks of the host-side plan (no GPU): for random problem descriptions, the library's
validation (domino_workspace_size) accepts exactly the configurations the documented rules allow,
and for every accepted one the workspace layout it prints with DOMINO_LOG=1 places each buffer on a
1 KiB boundary, inside the reported total, without overlapping another buffer."""
import re

import numpy as np
import pytest

PASSES = {"fwd": 0, "bwd": 1, "stack": 2, "stack_bwd": 3, "fwd_fp8": 6}


@pytest.fixture(scope="module")
def dlib():
    from comm_overlap_gb300 import build, domino
    build.build()
    return domino


def rules_allow(c: dict, pass_: int) -> bool:
    """The documented validation rules, stated independently of the library."""
    M, h, F, t, p, q = c["M"], c["h"], c["ffn"], c["t"], c["p"], c["q"]
    if M < 0 or h <= 0 or F <= 0 or t < 1 or p < 1 or q < 1:
        return False
    if M % p or h % q or F % t:
        return False
    Fi = F // t
    if h % 8 or Fi % 8 or (h // q) % 8:
        return False
    if pass_ == 6 and (h % 16 or Fi % 16):
        return False
    if M > 2**31 - 1 or h > 2**20 or F > 2**24:
        return False
    if (M // p) * ((h // q) // 8) >= 2**31:
        return False
    if pass_ in (2, 3) and c["layers"] < 1:
        return False
    return True


def random_cfg(rng):
    t = int(rng.choice([1, 2, 3, 4, 8, 16]))
    p = int(rng.choice([1, 2, 3, 4, 8]))
    q = int(rng.choice([1, 2, 4, 8]))
    # mostly valid sizes, with some broken divisibility or alignment
    m = int(rng.integers(0, 300)) * int(rng.choice([1, 8, 64]))
    M = m * p + (int(rng.integers(1, p)) if p > 1 and rng.random() < 0.15 else 0)
    h = 8 * q * int(rng.integers(1, 96)) + (int(rng.choice([4, 2, 8 * q + 8])) if rng.random() < 0.15 else 0)
    Fi = 8 * int(rng.integers(1, 200)) + (4 if rng.random() < 0.1 else 0)
    F = Fi * t + (1 if rng.random() < 0.1 else 0)
    return dict(M=M, h=h, ffn=F, t=t, p=p, q=q, act=int(rng.choice([2, 3])), sched=int(rng.integers(0, 4)),
                layers=int(rng.integers(1, 4)))


PLAN = re.compile(r"workspace=(\d+) B \[h@(\d+) ln@(\d+) dz@(\d+) hb@(\d+) gn@(\d+) qkv@(\d+) o@(\d+) "
                  r"partials@(\d+)\]")


def fused_split_bytes(m, n, t, units=76):
    tiles = -(-m // 256) * -(-n // 256)
    if tiles == 0 or t < 2:
        return 0
    u = min(tiles * t, units) if tiles < units else units
    rest = tiles % u
    if rest == 0 or u // rest < 2:
        return 0
    return rest * t * (256 * 256 * 4 + 4)


def buffers(c, pass_, off, total):
    """(name, offset, size) of each buffer the pass uses, from the documented layout."""
    M, h, F, t, p, q = c["M"], c["h"], c["ffn"], c["t"], c["p"], c["q"]
    m, n = M // p, h // q
    gated = c["act"] in (3, 4)
    a_rows = 2 * F if gated else F
    fused = c["sched"] == 3
    # the fused schedule keeps its shard sums on chip; it needs only the scratch of the shard split
    # of its last round of tiles (partial slots for the 76 CTA pairs of a GB300, then counters)
    if fused:
        slots, part = 1, fused_split_bytes(m, n, t)
    else:
        slots, part = (1 if p * q < 2 else 2), t * m * n * 4
    out = []
    if pass_ in (0, 2):
        out.append(("h", off["h"], m * F * 2))
        if pass_ == 2:
            out.append(("ln", off["ln"], m * h * 2))
    elif pass_ == 6:
        out.append(("h", off["h"], m * F))
    else:
        out.append(("dz", off["dz"], m * a_rows * 2))
        out.append(("hb", off["hb"], m * F * 2))
        if pass_ == 3:
            out.append(("gn", off["gn"], M * h * 2))
    up = (part + 1023) // 1024 * 1024
    for s in range(slots):
        out.append((f"part{s}", off["partials"] + s * up, part))
    return out


@pytest.mark.parametrize("pname", list(PASSES))
def test_random_plans_validate_and_lay_out(dlib, pname, capfd, monkeypatch):
    monkeypatch.setenv("DOMINO_LOG", "1")
    pass_ = PASSES[pname]
    rng = np.random.default_rng(1000 + pass_)
    accepted = 0
    for _ in range(120):
        c = random_cfg(rng)
        cfg = dlib.make_cfg(**c)
        capfd.readouterr()
        try:
            total = dlib.domino_workspace_size(cfg, pass_)
            ok = True
        except dlib.DominoError:
            ok = False
        assert ok == rules_allow(c, pass_), (pname, c)
        if not ok:
            continue
        err = capfd.readouterr().err
        if c["M"] == 0:
            assert total == 0
            continue
        accepted += 1
        mt = PLAN.search(err)
        assert mt, err
        assert int(mt.group(1)) == total
        off = dict(zip(["h", "ln", "dz", "hb", "gn", "qkv", "o", "partials"], map(int, mt.groups()[1:])))
        regions = buffers(c, pass_, off, total)
        for name, o, size in regions:
            assert o % 1024 == 0, (name, o)
            assert o + size <= total, (name, o, size, total)
        spans = sorted((o, o + size, name) for name, o, size in regions if size > 0)
        for (a0, a1, an), (b0, b1, bn) in zip(spans, spans[1:]):
            assert a1 <= b0, (pname, c, an, bn)
    assert accepted >= 20, accepted
