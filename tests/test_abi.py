"""C-ABI checks that need no GPU: the library builds and loads, exports every function
include/domino.h declares, and its host-only logic (validation, workspace sizing) behaves."""
import ctypes
import os
import re

import pytest

from conftest import ROOT

HEADER = os.path.join(ROOT, "include", "domino.h")


@pytest.fixture(scope="module")
def dlib():
    from comm_overlap_gb300 import build, domino
    build.build()
    return domino


def declared_functions():
    text = open(HEADER, encoding="utf-8").read()
    return sorted(set(re.findall(r"^DOMINO_API\s+[\w\s\*]+?\b(domino_\w+)\s*\(", text, flags=re.M)))


def test_header_declares_the_path_calls():
    names = declared_functions()
    for need in ("domino_create", "domino_destroy", "domino_workspace_size", "domino_mlp_fwd", "domino_mlp_bwd",
                 "domino_stack_fwd", "domino_shard_sum", "domino_status_string", "domino_last_error"):
        assert need in names


def test_library_exports_every_declared_symbol(dlib):
    lib = ctypes.CDLL(dlib.LIB_PATH)
    missing = [n for n in declared_functions() if not hasattr(lib, n)]
    assert not missing, missing
    # and the binding knows every one of them
    assert sorted(dlib._SIGS) == declared_functions()


def test_status_strings(dlib):
    for code, name in dlib.STATUS.items():
        assert dlib.domino_status_string(code) == name


def ws(dlib, **kw):
    return dlib.domino_workspace_size(dlib.make_cfg(**kw), dlib.PASS_FWD)


def test_workspace_size_formula(dlib):
    # forward: H (m x F bf16) + 2 partial slots of t x m x n fp32, each 1 KiB aligned
    def up(x):
        return (x + 1023) // 1024 * 1024
    M, h, F, t, p, q = 16384, 2560, 10240, 8, 2, 1
    m, n = M // p, h // q
    got = ws(dlib, M=M, h=h, ffn=F, t=t, p=p, q=q)
    assert got == up(m * F * 2) + 2 * up(t * m * n * 4)
    # one chunk only -> one slot
    got1 = ws(dlib, M=M, h=h, ffn=F, t=t, p=1, q=1)
    assert got1 == up(M * F * 2) + up(t * M * h * 4)
    # backward: dZ (m x 2F) + H (m x F) + slots
    cfg = dlib.make_cfg(M=32768, h=4096, ffn=14336, t=8, p=2, q=1, act=dlib.ACT_SWIGLU)
    m = 16384
    assert dlib.domino_workspace_size(cfg, dlib.PASS_BWD) == up(m * 2 * 14336 * 2) + up(m * 14336 * 2) + 2 * up(
        8 * m * 4096 * 4)
    # stack adds the LayerNorm buffer
    cfg = dlib.make_cfg(M=32768, h=4096, ffn=16384, t=4, p=2, q=2, layers=4)
    m, n = 16384, 2048
    assert dlib.domino_workspace_size(cfg, dlib.PASS_STACK) == up(m * 16384 * 2) + up(m * 4096 * 2) + 2 * up(
        4 * m * n * 4)
    # the fused schedule keeps its sums on chip: no partial slots, only the scratch of the shard
    # split of a short last round of tiles (256 KiB + a counter per shard of each of its tiles, for
    # the 76 CTA pairs of a GB300); 64 x 8 = 512 tiles leave 56 > 38 for the last round: none
    cfg = dlib.make_cfg(M=32768, h=4096, ffn=16384, t=4, p=2, q=2, layers=4, sched=dlib.SCHED_FUSED)
    assert dlib.domino_workspace_size(cfg, dlib.PASS_STACK) == up(m * 16384 * 2) + up(m * 4096 * 2)
    # GPT-3 2.7B: 32 x 10 = 320 tiles, 16 in the last round, 8 shards each
    M, h, F, t, p, q = 16384, 2560, 10240, 8, 2, 1
    m, n = M // p, h // q
    assert ws(dlib, M=M, h=h, ffn=F, t=t, p=p, q=q, sched=dlib.SCHED_FUSED) == up(m * F * 2) + up(
        16 * 8 * (256 * 256 * 4 + 4))
    # empty input needs nothing
    assert ws(dlib, M=0, h=64, ffn=64, t=2) == 0


@pytest.mark.parametrize("kw,status", [
    (dict(M=100, h=64, ffn=64, t=2, p=3), 1),      # M % p
    (dict(M=96, h=64, ffn=66, t=2), 3),            # F_i = 33 not a multiple of 8
    (dict(M=96, h=64, ffn=64, t=3), 1),            # F % t
    (dict(M=96, h=64, ffn=64, t=2, q=3), 1),       # h % q
    (dict(M=96, h=48, ffn=64, t=2, q=2), 3),       # h/q = 24 ok; make it fail below
    (dict(M=96, h=68, ffn=64, t=2), 3),            # h % 8
    (dict(M=96, h=64, ffn=64, t=0), 1),
    (dict(M=96, h=64, ffn=64, t=2, act=9), 1),
    (dict(M=96, h=64, ffn=64, t=2, sched=7), 1),
    (dict(M=96, h=64, ffn=64, t=2, flags=1), 1),
    (dict(M=96, h=64, ffn=64, t=2, reduce_ctas=-1), 1),
    (dict(M=96, h=64, ffn=64, t=2, attn_ctas=-1), 1),
    (dict(M=1 << 26, h=1 << 15, ffn=64, t=2), 2),  # m x n / 8 = 2^38 vectors in one reduction
])
def test_validation_errors(dlib, kw, status):
    if kw.get("h") == 48:
        # 48 / 2 = 24 is fine; 48 / 4 = 12 is not a multiple of 8
        kw = dict(kw, q=4)
    with pytest.raises(dlib.DominoError) as e:
        ws(dlib, **kw)
    assert e.value.status == status
    assert dlib.domino_last_error()


def test_stack_validation(dlib):
    cfg = dlib.make_cfg(M=64, h=64, ffn=64, t=2, layers=0)
    with pytest.raises(dlib.DominoError):
        dlib.domino_workspace_size(cfg, dlib.PASS_STACK)
    cfg = dlib.make_cfg(M=64, h=64, ffn=64, t=2, layers=2, ln_eps=0.0)
    with pytest.raises(dlib.DominoError):
        dlib.domino_workspace_size(cfg, dlib.PASS_STACK)


def test_shard_sum_host_validation(dlib):
    with pytest.raises(dlib.DominoError) as e:
        dlib.domino_shard_sum(0x1000, 2, 4, 12, None, 0, 0x2000, 16, stream=0)
    assert e.value.status == 3
    with pytest.raises(dlib.DominoError) as e:
        dlib.domino_shard_sum(0x1000, 0, 4, 16, None, 0, 0x2000, 16, stream=0)
    assert e.value.status == 1
    with pytest.raises(dlib.DominoError) as e:  # 2^31 16-byte vectors: beyond a 32-bit loop count
        dlib.domino_shard_sum(0x1000, 2, 1 << 20, 1 << 14, None, 0, 0x2000, 1 << 14, stream=0)
    assert e.value.status == 2


def test_create_without_gpu_fails_cleanly(dlib):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    with pytest.raises(dlib.DominoError) as e:
        dlib.domino_create()
    assert e.value.status in (5, 7)


def test_binding_refuses_missing_library(tmp_path, monkeypatch):
    from comm_overlap_gb300 import domino
    monkeypatch.setattr(domino, "_lib", None)
    monkeypatch.setattr(domino, "LIB_PATH", str(tmp_path / "nope.so"))
    with pytest.raises(domino.DominoError):
        domino.lib()


def test_plan_log(dlib, capfd, monkeypatch):
    """DOMINO_LOG=1 prints each validated plan (pass, sizes, schedule, workspace layout) to stderr;
    unset, nothing is printed."""
    cfg = dlib.make_cfg(M=512, h=256, ffn=512, t=2, p=2, q=1, sched=dlib.SCHED_INTRA)
    monkeypatch.delenv("DOMINO_LOG", raising=False)
    n = dlib.domino_workspace_size(cfg, dlib.PASS_FWD)
    assert "domino plan" not in capfd.readouterr().err
    monkeypatch.setenv("DOMINO_LOG", "1")
    assert dlib.domino_workspace_size(cfg, dlib.PASS_FWD) == n
    err = capfd.readouterr().err
    assert "domino plan: pass=fwd M=512 h=256 ffn=512 t=2 p=2 q=1 (chunk 256 x 256)" in err
    assert f"workspace={n} B" in err and "sched=intra" in err


def test_size_limits_are_exact(dlib):
    """The documented ranges are accepted up to their last value and refused one past it: at most
    2^31 - 1 tokens, and one reduction launch covering fewer than 2^31 16-byte vectors (m x n / 8)."""
    big = (1 << 31) - 1
    assert dlib.domino_workspace_size(dlib.make_cfg(M=big, h=8, ffn=8, t=1), dlib.PASS_FWD) > 0
    with pytest.raises(dlib.DominoError) as e:
        dlib.domino_workspace_size(dlib.make_cfg(M=big + 1, h=8, ffn=8, t=1), dlib.PASS_FWD)
    assert e.value.status == 2
    # m x n / 8 = (2^30 - 1) x 2 is the last count below 2^31; 2^30 x 2 is refused
    assert dlib.domino_workspace_size(dlib.make_cfg(M=(1 << 30) - 1, h=16, ffn=8, t=1), dlib.PASS_FWD) > 0
    with pytest.raises(dlib.DominoError) as e:
        dlib.domino_workspace_size(dlib.make_cfg(M=1 << 30, h=16, ffn=8, t=1), dlib.PASS_FWD)
    assert e.value.status == 2
    # a row split brings the same problem back under the reduction limit
    assert dlib.domino_workspace_size(dlib.make_cfg(M=1 << 30, h=16, ffn=8, t=1, p=2), dlib.PASS_FWD) > 0
