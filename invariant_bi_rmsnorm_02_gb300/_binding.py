"""placeholder until the C ABI exists"""
def load():
    raise RuntimeError("libbi.so not built")
