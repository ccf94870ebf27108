"""Loader for the worked layout examples in ``tests/golden/layout_examples.txt``."""
import os

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "layout_examples.txt")


def records():
    out = []
    with open(GOLDEN) as f:
        for lineno, line in enumerate(f, 1):
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            fields = line.split("|")
            out.append((lineno, fields[0], fields[1:]))
    return out


def parse_coord(text):
    """'5' -> 5, '(1,5)' -> (1, 5), '(1,(1,2))' -> (1, (1, 2))."""
    text = text.strip()
    if not text.startswith("("):
        return int(text)
    return eval(text, {"__builtins__": {}}, {})  # digits, commas and parentheses only


def ints(text):
    return [int(x) for x in text.split()]
