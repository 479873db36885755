"""Rules of the repository that are easy to break by accident (no GPU).

* The product package never imports the oracle: the oracle is test
  infrastructure, and the GPU path has no CPU fallback through it.
* No committed source reads, imports or runs anything under `_work/`.
* Every ncu command recorded under `profiles/` leaves the GPU clocks alone
  (`--clock-control none`).
"""

import os
import re

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PKG = os.path.join(ROOT, "block_diffusion_speculative_gather_gb300")
SOURCE_EXT = (".py", ".cu", ".cuh", ".h", ".c", ".cpp")


def _files(top, exts):
    for d, dirs, names in os.walk(top):
        dirs[:] = [x for x in dirs if x not in ("_build", "__pycache__", "_work", "gpurun_out",
                                                ".git", "baseline")]
        for n in names:
            if n.endswith(exts):
                yield os.path.join(d, n)


def test_product_package_never_imports_the_oracle():
    pat = re.compile(r"^\s*(from\s+oracle\b|import\s+oracle\b)|dflash_oracle", re.M)
    offenders = [p for p in _files(PKG, (".py",)) if pat.search(open(p).read())]
    assert not offenders, offenders


def test_no_committed_source_uses_the_scratch_folder():
    me = os.path.abspath(__file__)
    offenders = [p for p in _files(ROOT, SOURCE_EXT)
                 if os.path.abspath(p) != me and "_work/" in open(p, errors="ignore").read()]
    assert not offenders, offenders


def _commands(text):
    """Indented command blocks of a Markdown summary, continuation lines
    (trailing backslash) joined."""
    out, cur = [], ""
    for line in text.splitlines():
        if line.startswith("    ") and line.strip():
            cur += " " + line.strip().rstrip("\\")
            if not line.rstrip().endswith("\\"):
                out.append(cur)
                cur = ""
        elif cur:
            out.append(cur)
            cur = ""
    if cur:
        out.append(cur)
    return out


def test_profiled_ncu_commands_keep_the_clocks():
    seen = 0
    for p in _files(os.path.join(ROOT, "profiles"), (".md", ".txt")):
        for cmd in _commands(open(p).read()):
            for part in re.split(r"&&|;", cmd):
                words = part.split()
                # an ncu invocation: the word itself, possibly after env assignments
                lead = [w for w in words if "=" not in w][:1]
                if lead == ["ncu"]:
                    seen += 1
                    assert "--clock-control none" in part, (p, part)
    assert seen >= 4
