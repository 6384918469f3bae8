"""The C-ABI library builds, loads and exports every function the header declares; host-side
argument validation answers without touching a GPU."""
import ctypes
import os
import re
import subprocess

import pytest

import speculative_decoding_verification_spec_gb300 as sv
from speculative_decoding_verification_spec_gb300 import build_ext

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "spec_verify.h")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^[a-z_ ]+?[\s\*]+([a-z_]+)\s*\(", text, flags=re.M)))


@pytest.fixture(scope="module")
def lib():
    build_ext.build()
    return sv.load()


def test_header_declares_the_three_verify_calls():
    names = declared_functions()
    for n in ("spec_verify", "spec_verify_topk", "tree_verify_greedy", "spec_workspace_bytes",
              "spec_status_string"):
        assert n in names
    assert set(names) == set(sv.EXPORTS)


def test_library_exports_every_declared_symbol(lib):
    out = subprocess.run(["nm", "-D", "--defined-only", build_ext.LIB], capture_output=True,
                         text=True, check=True).stdout
    exported = {line.split()[-1] for line in out.splitlines() if line.strip()}
    for name in declared_functions():
        assert name in exported, name
        assert hasattr(lib, name)


def test_workspace_bytes(lib):
    a = sv.workspace_bytes(64, 5, 128256)
    assert a > 0 and a % 256 == 0
    assert sv.workspace_bytes(128, 5, 128256) >= a
    assert sv.workspace_bytes(64, 5, 128256, 50) > a
    assert sv.workspace_bytes(32, 0, 128256, 0, 64) > 0
    assert lib.spec_workspace_bytes(-1, 5, 10, 0, 0) == 0
    assert lib.spec_workspace_bytes(1, 5, 0, 0, 0) == 0


def test_host_validation_without_gpu(lib):
    P = ctypes.c_void_p
    fake = P(0x10000)  # never dereferenced: validation fails first
    ws = P(0x20000)
    INVALID, WORKSPACE = 1, 3

    def sv_call(B=2, gamma=3, V=100, T=1.0, dtype=1, target=fake, draft=fake, tok=fake, u=fake,
                acc=fake, out=fake, wsp=ws, wsb=1 << 30, topk=None):
        args = [target, draft, dtype, tok, u, B, gamma, V, T]
        tail = [acc, out, None, None, None, None, wsp, wsb, None]
        if topk is None:
            return lib.spec_verify(*args, *tail)
        return lib.spec_verify_topk(*args, topk, *tail)

    assert sv_call(B=0) == 0
    assert sv_call(B=-1) == INVALID
    assert sv_call(gamma=-1) == INVALID
    assert sv_call(V=0) == INVALID
    assert sv_call(T=0.0) == INVALID
    assert sv_call(T=float("nan")) == INVALID
    assert sv_call(T=float("inf")) == INVALID
    assert sv_call(T=1e-45) == INVALID
    assert sv_call(dtype=7) == INVALID
    assert sv_call(target=None) == INVALID
    assert sv_call(draft=None) == INVALID
    assert sv_call(u=None) == INVALID
    assert sv_call(out=None) == INVALID
    assert sv_call(target=P(0x10001)) == INVALID       # bf16 needs 2-byte alignment
    assert sv_call(wsp=None) == WORKSPACE
    assert sv_call(wsp=P(0x20008)) == WORKSPACE       # 16-byte alignment
    assert sv_call(wsb=16) == WORKSPACE
    assert sv_call(topk=0) == INVALID
    assert sv_call(topk=101) == INVALID
    assert lib.tree_verify_greedy(fake, 1, fake, fake, 2, 4, 10, 0, fake, fake, None, None, ws,
                                  1 << 30, None) == INVALID
    assert lib.tree_verify_greedy(fake, 1, None, fake, 2, 4, 10, 5, fake, fake, None, None, ws,
                                  1 << 30, None) == INVALID
    assert lib.tree_verify_greedy(fake, 1, fake, fake, 2, 4, 10, 5, fake, fake, None, None, ws,
                                  64, None) == WORKSPACE
    # tree_verify_sample: sizes, temperature, pointers and capacity, before any CUDA call
    F = ctypes.c_float

    def ts_call(B=2, N=4, Nq=5, V=1000, T=1.0, dtype=1, target=fake, draft=fake, par=fake,
                tok=fake, qr=fake, u=fake, max_out=5, acc=fake, out=fake):
        return lib.tree_verify_sample(target, draft, dtype, par, tok, qr, u, B, N, Nq, V, F(T),
                                      max_out, acc, out, None, None, None, None)

    assert ts_call(B=0) == 0
    for bad in (dict(B=-1), dict(N=-1), dict(Nq=-1), dict(V=0), dict(max_out=0), dict(T=0.0),
                dict(T=float("nan")), dict(dtype=3), dict(target=None), dict(draft=None),
                dict(Nq=0), dict(par=None), dict(tok=None), dict(qr=None), dict(u=None),
                dict(acc=None), dict(out=None), dict(target=P(0x10001)), dict(N=4097),
                dict(V=262145), dict(dtype=0, V=131073), dict(u=P(0x10002))):
        assert ts_call(**bad) == INVALID, bad
    # smc_verify: groups, particles, threshold and pointers, before any CUDA call
    def smc_call(G=2, Np=4, K=3, V=1000, T=1.0, eta=2.0, lw=fake, lwo=fake, u=fake, acc=fake,
                 out=fake, wsp=ws):
        return lib.smc_verify(fake, fake, 1, fake, lw, u, G, Np, K, V, F(T), F(eta), acc, out, lwo,
                              None, None, None, None, None, wsp, 1 << 30, None)

    assert smc_call(G=0) == 0
    for bad in (dict(G=-1), dict(Np=0), dict(Np=4097), dict(eta=float("nan")), dict(lw=None),
                dict(lwo=None), dict(T=0.0), dict(V=0), dict(K=-1), dict(u=None), dict(acc=None),
                dict(out=None), dict(lw=P(0x10002))):
        assert smc_call(**bad) == INVALID, bad
    assert smc_call(wsp=None) == WORKSPACE
    # spec_verify_greedy: sizes and pointers
    assert lib.spec_verify_greedy(fake, 1, fake, 0, 5, 100, fake, fake, None, ws, 1 << 30, None) == 0
    assert lib.spec_verify_greedy(fake, 1, fake, 2, -1, 100, fake, fake, None, ws, 1 << 30, None) == INVALID
    assert lib.spec_verify_greedy(fake, 1, None, 2, 3, 100, fake, fake, None, ws, 1 << 30, None) == INVALID
    assert lib.spec_verify_greedy(fake, 9, fake, 2, 3, 100, fake, fake, None, ws, 1 << 30, None) == INVALID
    assert lib.spec_verify_greedy(fake, 1, fake, 2, 3, 100, fake, fake, None, ws, 16, None) == WORKSPACE
    assert lib.spec_status_string(0) == b"ok"
    # tree_verify_typical: sizes, temperature, thresholds and pointers
    def ty_call(B=2, N=4, V=1000, T=1.0, eps=0.09, delta=0.3, par=fake, tok=fake, u=fake, wsp=ws,
                mo=5):
        return lib.tree_verify_typical(fake, 1, par, tok, u, B, N, V, F(T), F(eps), F(delta), mo,
                                       fake, fake, None, None, None, None, wsp, 1 << 30, None)

    assert ty_call(B=0) == 0
    for bad in (dict(B=-1), dict(N=-1), dict(N=2049), dict(V=0), dict(T=0.0), dict(eps=-1.0),
                dict(delta=float("inf")), dict(eps=float("nan")), dict(par=None), dict(tok=None),
                dict(u=None), dict(mo=0), dict(u=P(0x10002))):
        assert ty_call(**bad) == INVALID, bad
    assert ty_call(wsp=None) == WORKSPACE
    # spec_verify_topp: top_p > 0 and not NaN
    def tp_call(B=2, top_p=0.9):
        return lib.spec_verify_topp(fake, fake, 1, fake, fake, B, 3, 100, F(1.0), F(top_p), fake,
                                    fake, None, None, None, None, ws, 1 << 30, None)

    assert tp_call(B=0) == 0
    for bad in (dict(top_p=0.0), dict(top_p=-0.5), dict(top_p=float("nan")), dict(B=-1)):
        assert tp_call(**bad) == INVALID, bad
    # spec_verify_masked: the mask is required (B > 0) and 4-byte aligned
    def mk_call(B=2, mask=fake):
        return lib.spec_verify_masked(fake, fake, 1, fake, fake, mask, B, 3, 100, F(1.0), fake, fake,
                                      None, None, None, None, ws, 1 << 30, None)

    assert mk_call(B=0, mask=None) == 0
    assert mk_call(mask=None) == INVALID
    assert mk_call(mask=P(0x10002)) == INVALID
    assert mk_call(B=-1) == INVALID
    # the no-allocation entry point refuses oversized or invalid sizes before any CUDA call
    TOO_LARGE = 4
    assert lib.spec_verify_noalloc(fake, fake, 1, fake, fake, 1024, 7, 152064, 1.0, fake, fake,
                                   None, None, None, None, None) == TOO_LARGE
    assert lib.spec_verify_noalloc(fake, fake, 1, fake, fake, 2, 3, 0, 1.0, fake, fake,
                                   None, None, None, None, None) == INVALID


def test_no_cpu_fallback_in_the_binding():
    import torch
    x = torch.zeros(1, 2, 8)
    with pytest.raises(sv.SpecVerifyError):
        sv.spec_verify(x, x[:, :1], torch.zeros(1, 1, dtype=torch.int32),
                       torch.zeros(1, 3), 1.0)
