"""The usage example in README.md runs as written (its one python block), and its
outputs have the documented shapes and no device-side failure."""
import os

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_readme_example_runs(cuda_dev):
    with open(os.path.join(ROOT, "README.md")) as f:
        text = f.read()
    start = text.index("```python\n") + len("```python\n")
    code = text[start:text.index("```", start)]
    scope = {}
    exec(compile(code, "README.md", "exec"), scope)
    torch = scope["torch"]
    torch.cuda.synchronize()
    assert tuple(scope["y"].shape) == (16384, 2048)
    assert tuple(scope["y_slots"].shape) == (16384, 8, 2048)
    assert tuple(scope["out"].shape) == (16384, 2048)
    assert tuple(scope["dx"].shape) == (16384, 2048)
    assert tuple(scope["y_mx"].shape) == (16384, 2048)
    assert scope["situ"].device_status(clear=True) == 0
