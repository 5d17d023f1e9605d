"""The product path has no fallback: without libdm.so every call raises, and
the package never imports, links or reads the FP64 oracle."""
import os
import re
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PKG = os.path.join(ROOT, "fp8_attention_gb300")


def run_child(code: str) -> subprocess.CompletedProcess:
    return subprocess.run([sys.executable, "-c", code], cwd=ROOT, capture_output=True, text=True,
                          timeout=300)


def test_calls_raise_when_the_library_is_missing(tmp_path):
    missing = str(tmp_path / "libdm.so")
    code = f"""
import fp8_attention_gb300 as dm
dm.LIB_PATH = {missing!r}
dm._lib = None
for call in (dm.dm_version, lambda: dm.dm_status_string(0), lambda: dm.dm_set_knob(0, 1)):
    try:
        call()
    except RuntimeError as e:
        assert "missing" in str(e), e
    else:
        raise SystemExit("a call returned without the library")
print("raised")
"""
    r = run_child(code)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "raised" in r.stdout


def test_package_does_not_import_the_oracle():
    r = run_child("import sys, fp8_attention_gb300, fp8_attention_gb300.inputs\n"
                  "print(sorted(m for m in sys.modules if m == 'oracle' or m.startswith('oracle.')))")
    assert r.returncode == 0, r.stdout + r.stderr
    assert r.stdout.strip() == "[]", r.stdout


def test_package_sources_never_name_the_oracle():
    pattern = re.compile(r"\boracle\b|liboracle")
    hits = []
    for dirpath, _, files in os.walk(PKG):
        if "__pycache__" in dirpath:
            continue
        for f in files:
            if not f.endswith((".py", ".cu", ".cuh", ".h", ".cpp")):
                continue
            path = os.path.join(dirpath, f)
            for n, line in enumerate(open(path, encoding="utf-8"), 1):
                if pattern.search(line) and ("import" in line or "CDLL" in line or "load" in line):
                    hits.append(f"{os.path.relpath(path, ROOT)}:{n}: {line.strip()}")
    assert not hits, "\n".join(hits)
