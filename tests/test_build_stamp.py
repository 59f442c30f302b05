"""The library build's up-to-date rule (CPU only; the compiler is faked):
a stamp of the flags and source contents decides, so rewritten files with
unchanged contents do not trigger a compile, changed contents do, and with
no stamp the source times decide."""
import os
import time

from selective_state_space_113_b300 import build as libbuild


def _setup(tmp_path, monkeypatch):
    srcs = []
    for name in ("a.cuh", "api.cu"):
        p = tmp_path / name
        p.write_text(f"// {name}\n")
        srcs.append(str(p))
    out = str(tmp_path / "libfake.so")
    stamp = str(tmp_path / "stamp" / "libfake.so.stamp")
    compiles = []

    def fake_run(cmd, check):
        compiles.append(cmd)
        with open(cmd[cmd.index("-o") + 1], "wb") as fh:
            fh.write(b"\x7fELF")

    monkeypatch.setattr(libbuild, "sources", lambda: srcs)
    monkeypatch.setattr(libbuild, "stamp_path", lambda o=out: stamp)
    monkeypatch.setattr(libbuild, "nvcc_path", lambda: "nvcc")
    monkeypatch.setattr(libbuild.subprocess, "run", fake_run)
    return srcs, out, stamp, compiles


def _touch_later(path):
    t = time.time() + 5
    os.utime(path, (t, t))


def test_stamp_decides(tmp_path, monkeypatch):
    srcs, out, stamp, compiles = _setup(tmp_path, monkeypatch)
    libbuild.build(out)
    assert len(compiles) == 1 and os.path.exists(stamp)
    libbuild.build(out)
    assert len(compiles) == 1                      # current: nothing to do
    _touch_later(srcs[0])
    libbuild.build(out)
    assert len(compiles) == 1                      # newer time, same contents
    with open(srcs[0], "a") as fh:
        fh.write("// changed\n")
    libbuild.build(out)
    assert len(compiles) == 2                      # changed contents
    libbuild.build(out, extra=("-DX",))
    assert len(compiles) == 3                      # extra flags always compile
    libbuild.build(out, force=True)
    assert len(compiles) == 4


def test_without_stamp_times_decide(tmp_path, monkeypatch):
    srcs, out, stamp, compiles = _setup(tmp_path, monkeypatch)
    with open(out, "wb") as fh:
        fh.write(b"\x7fELF")
    t = time.time() + 10
    os.utime(out, (t, t))
    assert libbuild.up_to_date(out)                # older sources, no stamp
    t2 = time.time() + 20
    os.utime(srcs[1], (t2, t2))
    assert not libbuild.up_to_date(out)
    libbuild.build(out)
    assert len(compiles) == 1 and os.path.exists(stamp)
