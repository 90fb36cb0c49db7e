"""Readers for the hand-written fixtures under tests/golden/ (plain text, cited in each file)."""
import os

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def lines(name):
    with open(os.path.join(GOLDEN, name)) as f:
        for raw in f:
            s = raw.strip()
            if s and not s.startswith("#"):
                yield s


def ints(field):
    field = field.strip()
    return [] if field == "-" else [int(v) for v in field.split()]


def route_cases():
    names = {"FOLD": 0, "SKIP": 1, "REFUSE": 2}
    for s in lines("route_truth.txt"):
        slot, active, has, exp = s.split()
        yield int(slot), int(active), int(has), names[exp]


def decode_map_cases():
    for s in lines("decode_map.txt"):
        slots, padded, active, has, exp = s.split("|")
        yield ints(slots), int(padded), int(active), int(has), ints(exp)


def host_map_cases():
    for s in lines("host_map.txt"):
        cu, slots, exp = s.split("|")
        yield ints(cu), ints(slots), (None if exp.strip() == "NONE" else ints(exp))


def pack_cases():
    for s in lines("pack.txt"):
        parts = [p.strip() for p in s.split("|")]
        entries = []
        if parts[0] != "-":
            for ent in parts[0].split(","):
                i, a, b, sc = ent.split(":")
                entries.append((int(i), int(a), int(b), float(sc)))
        if parts[1] == "EMPTY":
            yield entries, None
            continue
        yield entries, (int(parts[1]), [int(v) for v in parts[2].split()],
                        [int(v) for v in parts[3].split()], [float(v) for v in parts[4].split()])


def window_cases():
    for s in lines("windows.txt"):
        head, tail = s.split("|")
        total, cap = (int(v) for v in head.split())
        tail = tail.strip()
        if tail == "PANIC":
            yield total, cap, "PANIC"
        elif tail == "-":
            yield total, cap, []
        else:
            yield total, cap, [tuple(int(v) for v in w.split(":")) for w in tail.split()]


def wc_cases():
    for s in lines("wc.txt"):
        a, b, m, e = (int(v) for v in s.split())
        yield a, b, m, e
