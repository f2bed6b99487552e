"""libps from plain C: the header compiles as strict C99, and a C program that
uses only include/ps.h and the CUDA runtime (tests/c_abi/round.c) runs one
round (scoring, suffix sums, log A and the walk; PreSTO section 3.2 steps
(2)-(3)) with results equal to the Python binding's and within the parity
tolerances of the oracle's.
"""

import os
import shutil
import subprocess

import numpy as np
import pytest
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CUDA_HOME = os.environ.get("CUDA_HOME", "/usr/local/cuda")
SRC = os.path.join(ROOT, "tests", "c_abi", "round.c")
LIBDIR = os.path.join(ROOT, "mh_prefetch_subtree_gb300")


def _gcc():
    gcc = shutil.which("gcc")
    if gcc is None:
        pytest.skip("gcc is not installed")
    return gcc


def _build_lib():
    import __graft_entry__
    __graft_entry__.build()


def _build_round(out_dir) -> str:
    _build_lib()
    exe = os.path.join(str(out_dir), "round")
    cmd = [_gcc(), "-std=c99", "-O2", "-Wall", "-Wextra", "-Werror",
           "-I", os.path.join(ROOT, "include"), "-I", os.path.join(CUDA_HOME, "include"),
           SRC, "-o", exe, "-L", LIBDIR, "-lps", "-L", os.path.join(CUDA_HOME, "lib64"),
           "-lcudart", "-Wl,-rpath," + LIBDIR + ":" + os.path.join(CUDA_HOME, "lib64")]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    return exe


def test_header_is_plain_c99(tmp_path):
    src = tmp_path / "use_ps.c"
    src.write_text('#include "ps.h"\n'
                   "int main(void) { ps_subtree_batch b; ps_tree t; (void)b; (void)t;\n"
                   "  return ps_version() == 0; }\n")
    r = subprocess.run([_gcc(), "-std=c99", "-pedantic", "-Wall", "-Wextra", "-Werror",
                        "-I", os.path.join(ROOT, "include"), "-c", str(src), "-o",
                        str(tmp_path / "use_ps.o")], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr


def test_c_caller_builds_and_links(tmp_path):
    if not os.path.exists(os.path.join(CUDA_HOME, "include", "cuda_runtime_api.h")):
        pytest.skip("CUDA runtime headers not found")
    assert os.path.exists(_build_round(tmp_path))


def _write_inputs(w, d):
    """The batch and tree of workload w as the raw files round.c reads."""
    from oracle.hostcopy import logits_np
    lay = w.layout
    os.makedirs(d, exist_ok=True)
    lg, dt = logits_np(w.logits)
    dtype = 0 if dt == "bf16" else 1
    meta = (f"{w.V} {lay.T} {dtype} {lay.n_chains} {lay.n_seg} {lay.n_rows} "
            f"{len(lay.acc)} {w.max_steps} {lg.shape[1]} {w.alpha!r} {w.tau!r}\n")
    with open(os.path.join(d, "meta.txt"), "w") as f:
        f.write(meta)
    np.ascontiguousarray(lg).tofile(os.path.join(d, "logits.bin"))
    w.tokens.cpu().numpy().astype(np.int32).tofile(os.path.join(d, "tokens.bin"))
    for name in ("chain_seg0", "seg_cut", "seg_src", "chain_node0", "acc", "rej", "req"):
        np.asarray(getattr(lay, name), dtype=np.int32).tofile(os.path.join(d, name + ".bin"))
    np.asarray(lay.seg_row0, dtype=np.int64).tofile(os.path.join(d, "seg_row0.bin"))
    np.asarray(w.u, dtype=np.float64).tofile(os.path.join(d, "u.bin"))


def _read_outputs(d, w):
    lay = w.layout
    g = {k: np.fromfile(os.path.join(d, k + ".bin"), dtype=np.float64)
         for k in ("lp0", "lq", "log_ratio", "log_accept")}
    for k in ("state_seg", "end_node", "k_delta", "path"):
        g[k] = np.fromfile(os.path.join(d, k + ".bin"), dtype=np.int32)
    with open(os.path.join(d, "status.txt")) as f:
        g["status"], g["wstatus"] = (int(x) for x in f.read().split())
    assert g["lp0"].shape == (lay.n_rows,) and g["path"].shape == (
        lay.n_chains * (w.max_steps + 1),)
    return g


@pytest.mark.gpu
@pytest.mark.parametrize("case", ["config1", "config2_small"])
def test_c_caller_round_matches_the_binding_and_the_oracle(tmp_path, case):
    import mh_prefetch_subtree_gb300 as ps
    from synth import make_workload
    from tests import gpu_harness as H
    dev = torch.device("cuda:0")
    exe = _build_round(tmp_path)
    if case == "config1":
        w = make_workload(1, device=dev)
    else:
        w = make_workload(2, device=dev, T=48, n_pf=6, seed=61)
    _write_inputs(w, tmp_path / "in")
    os.makedirs(tmp_path / "out")
    r = subprocess.run([exe, str(tmp_path / "in"), str(tmp_path / "out")],
                       capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr
    assert r.stdout.startswith("libps")
    g = _read_outputs(tmp_path / "out", w)
    assert g["status"] == 0 and g["wstatus"] == 0, ps.dev_status_names(g["status"] | g["wstatus"])

    # the same round through the Python binding gives the same bits
    d = ps.DeviceSubtree.create(layout=w.layout, u=w.u, logits=w.logits, tokens=w.tokens,
                                V=w.V, alpha=w.alpha, tau=w.tau, max_steps=w.max_steps)
    d.step()
    torch.cuda.synchronize()
    for k in ("lp0", "lq", "log_ratio", "log_accept", "state_seg", "end_node", "k_delta",
              "path"):
        b = d.t[k].cpu().numpy()
        assert np.array_equal(g[k], b, equal_nan=np.issubdtype(b.dtype, np.floating)), k

    # and the oracle's values within the parity tolerances
    o = H.run_oracle(w)
    H.check_rows(g, o)
    H.check_log_accept(w, g, o)
    H.check_walk(w, g, o)
