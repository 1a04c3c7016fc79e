"""The usage example of the README runs as written."""
import os
import re

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_readme_usage_example_runs():
    text = open(os.path.join(ROOT, "README.md")).read()
    usage = text[text.index("## Usage"):]
    code = re.search(r"```python\n(.*?)```", usage, re.S).group(1)
    exec(compile(code, "README.md", "exec"), {})
