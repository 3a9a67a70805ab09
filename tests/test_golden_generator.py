"""The closed-form golden file is reproducible: its committed generator (40-digit decimal, no
import from the oracle or the package) writes exactly the committed text."""

import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
GEN = os.path.join(HERE, "golden", "make_closed_forms.py")


def test_generator_reproduces_closed_forms():
    r = subprocess.run([sys.executable, GEN, "--check"], capture_output=True, text=True)
    assert r.returncode == 0, r.stdout + r.stderr


def test_generator_imports_nothing_of_the_method():
    text = open(GEN).read()
    for name in ("oracle", "online_softmax_flashattention_gb300", "seeded_inputs", "numpy", "torch"):
        assert f"import {name}" not in text and f"from {name}" not in text, name
